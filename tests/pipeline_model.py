"""CPU model of the forward kernel's mbarrier protocol, for one CTA.

Every role of the kernel is a generator that yields the barrier waits and
arrivals it performs, in the kernel's order: the TMA producer, the two S
issuers, the two PV issuers and the softmax warps of both query tiles. A
random scheduler interleaves them with an in-order tensor pipe (commits fire
when they reach its head) and out-of-order TMA completions.

A barrier here counts completed phases. Waits name the completion they need;
the kernel passes only its parity, which is exact only while the barrier is
at most one phase past the awaited completion. ``Bar.done`` asserts exactly
that, so a protocol that lets a barrier run two phases ahead of a waiter
fails here even when the interleaving happens not to deadlock.

This models the kernel's synchronisation only (no data). Causal block counts
follow the kernel: 128-row query tiles, two per work item, 64-key blocks.
"""
import random

BQ, BK, ROWS = 128, 64, 256


class Bar:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.phase = name, count, count, 0

    def arrive(self, n=1):
        self.pending -= n
        assert self.pending >= 0, f"{self.name}: more arrivals than the phase expects"
        if self.pending == 0:
            self.phase += 1
            self.pending = self.count

    def done(self, index):
        assert index < 0 or self.phase <= index + 1, (
            f"{self.name}: waiting for completion {index} while the barrier is at phase {self.phase} "
            "(the parity wait would alias)")
        # a parity wait succeeds when the phase count's parity differs from the awaited one's: too
        # early if the barrier is an odd number of completions short of the awaited one
        assert index < 0 or self.phase >= index or not ((self.phase ^ index) & 1), (
            f"{self.name}: waiting for completion {index} while only {self.phase} completed "
            "(the parity wait would succeed early)")
        return self.phase > index


def tile_nkv(N, causal, q0, t):
    r0 = q0 + t * BQ
    if r0 >= N:
        return 0
    nkv = (N + BK - 1) // BK
    if not causal:
        return nkv
    return (min(N, r0 + BQ) - 1) // BK + 1


class Deadlock(AssertionError):
    pass


def simulate(N, causal, items, ring, seed, softmax_warps=4, per_buffer_p=True, rescale_prob=0.1,
             skip_empty_items=True, item_ring=0, ring_waits_empty=True):
    """Run one CTA's item list (first query rows) to completion; raise Deadlock or
    AssertionError on a protocol fault. ``per_buffer_p=False`` models a single
    P-ready barrier per tile (a protocol that is known to alias);
    ``skip_empty_items=False`` a producer that loads K block 0 even for an item
    with no rows (known to leave the K ring out of step).

    ``item_ring`` > 0 models the packed-batch kernel: a scheduler warp publishes
    each item, then an end marker, into a ring of that many slots (full barrier:
    one arrival; empty barrier: one arrival per consumer warp), and every role
    takes its items from the ring. ``ring_waits_empty=False`` is a scheduler
    that refills a slot without waiting for its readers (it must be caught)."""
    rnd = random.Random(seed)
    B = {}

    def bar(name, count):
        B[name] = Bar(name, count)

    for t in range(2):
        for name, c in (("q_full", 1), ("q_empty", 1), ("s_full", 1), ("s_free", BQ), ("pv_done0", 1),
                        ("pv_done1", 1)):
            bar(f"{name}{t}", c)
        if per_buffer_p:
            bar(f"p_full{t}0", BQ)
            bar(f"p_full{t}1", BQ)
        else:
            bar(f"p_full{t}", BQ)
    for s in range(ring):
        bar(f"k_full{s}", 1)
        bar(f"k_empty{s}", 2)
        bar(f"v_full{s}", 1)
        bar(f"v_empty{s}", 2)
    consumers = 5 + 2 * softmax_warps
    for s in range(item_ring):
        bar(f"item_full{s}", 1)
        bar(f"item_empty{s}", consumers)
    tensor_pipe, tma = [], []

    def take(i):
        # read list entry i (i == len(items) is the end marker) from the ring
        if item_ring:
            yield ("wait", f"item_full{i % item_ring}", i // item_ring)
            yield ("arrive", f"item_empty{i % item_ring}", 1)

    def scheduler():
        for i in range(len(items) + 1):
            if ring_waits_empty:
                yield ("wait", f"item_empty{i % item_ring}", i // item_ring - 1)
            yield ("arrive", f"item_full{i % item_ring}", 1)

    def p_full_name(t, g):
        return (f"p_full{t}{g & 1}", g >> 1) if per_buffer_p else (f"p_full{t}", g)

    def counts(q0):
        # an item is a first query row, or (first row, sequence length) in a packed batch, or
        # (first row, sequence length, row limit) for a single-tile unit of the dense schedule
        if isinstance(q0, int):
            q0, n_seq, nrow = q0, N, N
        elif len(q0) == 2:
            (q0, n_seq), nrow = q0, q0[1]
        else:
            q0, n_seq, nrow = q0
        n = [tile_nkv(n_seq, causal, q0, t) if q0 + t * BQ < nrow else 0 for t in range(2)]
        return n, max(n)

    def producer():
        qcount, kpos, vpos = [0, 0], 0, 0
        for i, q0 in enumerate(items):
            yield from take(i)
            n, nmax = counts(q0)
            for t in range(2):
                if n[t]:
                    yield ("wait", f"q_empty{t}", qcount[t] - 1)
                    tma.append(f"q_full{t}")
                    qcount[t] += 1
            order = (["K"] if nmax > 0 or not skip_empty_items else []) + [x for j in range(nmax)
                                                   for x in (["K"] if j + 1 < nmax else []) + ["V"]]
            for kind in order:
                if kind == "K":
                    yield ("wait", f"k_empty{kpos % ring}", kpos // ring - 1)
                    tma.append(f"k_full{kpos % ring}")
                    kpos += 1
                else:
                    yield ("wait", f"v_empty{vpos % ring}", vpos // ring - 1)
                    tma.append(f"v_full{vpos % ring}")
                    vpos += 1
        yield from take(len(items))

    def s_issuer(t):
        qcount = issued = kpos = 0
        for i, q0 in enumerate(items):
            yield from take(i)
            n, nmax = counts(q0)
            if n[t]:
                yield ("wait", f"q_full{t}", qcount)
                qcount += 1
            for j in range(nmax):
                s = kpos % ring
                yield ("wait", f"k_full{s}", kpos // ring)
                kpos += 1
                if j >= n[t]:
                    yield ("arrive", f"k_empty{s}", 1)
                    continue
                if issued:
                    yield ("wait", f"s_free{t}", issued - 1)
                issued += 1
                tensor_pipe.extend([("commit", f"s_full{t}")] + ([("commit", f"q_empty{t}")] if j == n[t] - 1 else [])
                                   + [("commit", f"k_empty{s}")])
        yield from take(len(items))

    def pv_issuer(t):
        g = vpos = 0
        for i, q0 in enumerate(items):
            yield from take(i)
            n, nmax = counts(q0)
            for j in range(nmax):
                s = vpos % ring
                yield ("wait", f"v_full{s}", vpos // ring)
                vpos += 1
                if j >= n[t]:
                    yield ("arrive", f"v_empty{s}", 1)
                    continue
                yield ("wait",) + p_full_name(t, g)
                tensor_pipe.extend([("commit", f"pv_done{t}{g & 1}"), ("commit", f"v_empty{s}")])
                g += 1
        yield from take(len(items))

    def softmax(t):
        scount = g = 0
        for i, q0 in enumerate(items):
            yield from take(i)
            n, _ = counts(q0)
            if not n[t]:
                continue
            for j in range(n[t]):
                yield ("wait", f"s_full{t}", scount)
                scount += 1
                yield ("arrive", f"s_free{t}", BQ // softmax_warps)
                if j > 0 and rnd.random() < rescale_prob:  # O rescale needs the previous product
                    yield ("wait", f"pv_done{t}{(g - 1) & 1}", (g - 1) >> 1)
                if g >= 2:  # P buffer g & 1 was last read by product g - 2
                    yield ("wait", f"pv_done{t}{g & 1}", (g - 2) >> 1)
                yield ("arrive", p_full_name(t, g)[0], BQ // softmax_warps)
                g += 1
            yield ("wait", f"pv_done{t}{(g - 1) & 1}", (g - 1) >> 1)  # epilogue
        yield from take(len(items))

    agents = {"producer": producer(), "S0": s_issuer(0), "S1": s_issuer(1), "PV0": pv_issuer(0),
              "PV1": pv_issuer(1)}
    if item_ring:
        agents["scheduler"] = scheduler()
    for t in range(2):
        for w in range(softmax_warps):
            agents[f"softmax{t}.{w}"] = softmax(t)
    waiting = {k: None for k in agents}
    while agents or tensor_pipe or tma:
        ready = [k for k in agents if waiting[k] is None or B[waiting[k][1]].done(waiting[k][2])]
        if tensor_pipe:
            ready.append("#tensor")
        if tma:
            ready.append("#tma")
        if not ready:
            raise Deadlock(f"deadlock: {[(k, waiting[k]) for k in agents]}")
        c = rnd.choice(ready)
        if c == "#tensor":
            _, name = tensor_pipe.pop(0)
            B[name].arrive(1)
            continue
        if c == "#tma":
            B[tma.pop(rnd.randrange(len(tma)))].arrive(1)
            continue
        try:
            while True:
                ev = next(agents[c])
                if ev[0] == "arrive":
                    B[ev[1]].arrive(ev[2])
                    continue
                waiting[c] = ev
                break
        except StopIteration:
            del agents[c]
            waiting[c] = None
    return True


def simulate_bwd(n_it, stages, seed, grad_warps=8):
    """The backward kernel's protocol for one CTA (one key block visiting n_it
    query blocks): TMA producer, MMA issuer, and the gradient warps (two
    warpgroups, 256 arrivals per phase on their barriers)."""
    rnd = random.Random(seed)
    B = {}
    n = 32 * grad_warps
    for name, c in (("kv", 1), ("sp_full", 1), ("p_full", n), ("dq_full", 1), ("dq_free", n), ("drain", 1),
                    ("stats", n)):
        B[name] = Bar(name, c)
    for s in range(stages):
        B[f"qd_full{s}"] = Bar(f"qd_full{s}", 1)
        B[f"qd_empty{s}"] = Bar(f"qd_empty{s}", 1)
    tensor_pipe, tma = [], []

    def producer():
        tma.append("kv")
        for it in range(n_it):
            s = it % stages
            yield ("wait", f"qd_empty{s}", it // stages - 1)
            tma.append(f"qd_full{s}")

    def mma():
        yield ("wait", "kv", 0)
        for it in range(n_it):
            s = it % stages
            yield ("wait", f"qd_full{s}", it // stages)
            if it > 0:
                yield ("wait", "dq_free", it - 1)
            tensor_pipe.append(("commit", "sp_full"))
            yield ("wait", "p_full", it)
            tensor_pipe.extend([("commit", "dq_full"), ("commit", f"qd_empty{s}")])
        tensor_pipe.append(("commit", "drain"))
        yield ("wait", "drain", 0)

    def grads():
        for it in range(n_it):
            yield ("arrive", "stats", 32)  # statistics of block it stored (their readers passed p_full(it-1))
            yield ("wait", "stats", it)
            yield ("wait", "sp_full", it)
            yield ("arrive", "p_full", 32)
            yield ("wait", "dq_full", it)
            yield ("arrive", "dq_free", 32)

    agents = {"producer": producer(), "mma": mma()}
    for w in range(grad_warps):
        agents[f"grads{w}"] = grads()
    waiting = {k: None for k in agents}
    while agents or tensor_pipe or tma:
        ready = [k for k in agents if waiting[k] is None or B[waiting[k][1]].done(waiting[k][2])]
        if tensor_pipe:
            ready.append("#tensor")
        if tma:
            ready.append("#tma")
        if not ready:
            raise Deadlock(f"deadlock: {[(k, waiting[k]) for k in agents]}")
        c = rnd.choice(ready)
        if c == "#tensor":
            B[tensor_pipe.pop(0)[1]].arrive(1)
            continue
        if c == "#tma":
            B[tma.pop(rnd.randrange(len(tma)))].arrive(1)
            continue
        try:
            while True:
                ev = next(agents[c])
                if ev[0] == "arrive":
                    B[ev[1]].arrive(ev[2])
                    continue
                waiting[c] = ev
                break
        except StopIteration:
            del agents[c]
            waiting[c] = None
    return True


def simulate_bwd_halves(n_it, stages, seed):
    """Protocol of the d = 64 backward kernel that overlaps the two 64-row halves
    of each query block: S/dP per half, dV/dK per half, the next block's S/dP
    issued between them, dQ of block i read out by the gradient warpgroups
    after their pass of block i + 1."""
    rnd = random.Random(seed)
    B = {}
    for name, c in (("kv", 1), ("dq_full", 1), ("dq_free", 256), ("drain", 1)):
        B[name] = Bar(name, c)
    for h in range(2):
        for name, c in (("sp_full", 1), ("p_full", 128), ("stats", 128)):
            B[f"{name}{h}"] = Bar(f"{name}{h}", c)
    for s in range(stages):
        B[f"qd_full{s}"] = Bar(f"qd_full{s}", 1)
        B[f"qd_empty{s}"] = Bar(f"qd_empty{s}", 1)
    tensor_pipe, tma = [], []

    def producer():
        tma.append("kv")
        for it in range(n_it):
            s = it % stages
            yield ("wait", f"qd_empty{s}", it // stages - 1)
            tma.append(f"qd_full{s}")

    def mma():
        # per block: dV,dK(A, i)  S,dP(A, i+1)  dV,dK(B, i)  S,dP(B, i+1)  dQ(i); the issuing warp
        # never waits for its own products (a warpgroup's wait for its next S covers them)
        yield ("wait", "kv", 0)
        yield ("wait", "qd_full0", 0)
        tensor_pipe.extend([("commit", "sp_full0"), ("commit", "sp_full1")])
        for it in range(n_it):
            nxt = it + 1 < n_it
            yield ("wait", "p_full0", it)
            if nxt:
                s1 = (it + 1) % stages
                yield ("wait", f"qd_full{s1}", (it + 1) // stages)
                tensor_pipe.append(("commit", "sp_full0"))
            yield ("wait", "p_full1", it)
            tensor_pipe.append(("commit", f"qd_empty{it % stages}"))
            if nxt:
                tensor_pipe.append(("commit", "sp_full1"))
            if it > 0:
                yield ("wait", "dq_free", it - 1)
            tensor_pipe.append(("commit", "dq_full"))
        tensor_pipe.append(("commit", "drain"))
        yield ("wait", "drain", 0)

    def grads(h):
        def readout(blk):
            yield ("wait", "dq_full", blk)
            yield ("arrive", "dq_free", 32)
        for it in range(n_it):
            yield ("arrive", f"stats{h}", 32)
            yield ("wait", f"stats{h}", it)
            yield ("wait", f"sp_full{h}", it)
            yield ("arrive", f"p_full{h}", 32)
            if it > 0:
                yield from readout(it - 1)
        yield from readout(n_it - 1)

    agents = {"producer": producer(), "mma": mma()}
    for h in range(2):
        for w in range(4):
            agents[f"g{h}.{w}"] = grads(h)
    waiting = {k: None for k in agents}
    while agents or tensor_pipe or tma:
        ready = [k for k in agents if waiting[k] is None or B[waiting[k][1]].done(waiting[k][2])]
        if tensor_pipe:
            ready.append("#tensor")
        if tma:
            ready.append("#tma")
        if not ready:
            raise Deadlock(f"deadlock: {[(k, waiting[k]) for k in agents]}")
        c = rnd.choice(ready)
        if c == "#tensor":
            B[tensor_pipe.pop(0)[1]].arrive(1)
            continue
        if c == "#tma":
            B[tma.pop(rnd.randrange(len(tma)))].arrive(1)
            continue
        try:
            while True:
                ev = next(agents[c])
                if ev[0] == "arrive":
                    B[ev[1]].arrive(ev[2])
                    continue
                waiting[c] = ev
                break
        except StopIteration:
            del agents[c]
            waiting[c] = None
    return True


def simulate_bk128(N, causal, items, rk, rv, seed, rescale_prob=0.1, item_ring=0, s_waits_free=True,
                   p_waits_pv=True, late_weight=1.0, pv_after_next_s=True, s_issued_barriers=2):
    """The 128-key-block forward (fa_fwd_bk128_kernel) for one CTA: TMA producer,
    the S issuer (S_t(j) for t = 0, 1 in turn into the one S buffer), one P V
    issuer per tile, the eight softmax warps and (``item_ring`` > 0) the
    packed-batch item list.

    Softmax warp w = 4 t + q handles the rows of TMEM lane quadrant q of tile t,
    all 128 keys of each block; the four warps of tile t copy out each of the
    tile's S products and release the S buffer.

    Besides the barrier checks of ``simulate`` the model tracks the S buffer and
    each tile's P buffer, so that an S product that overwrites an S the softmax
    has not copied out, a P stored over one its P V product has not read, or a
    softmax that reads the wrong S, fails here. The commits of P V products may
    reach their barriers late (measured on the GPU: several hundred cycles after
    later commits), in order among themselves (``late_weight`` < 1 delays them
    further); a P V product counts as done for O only when its commit arrives,
    and the softmax may rescale or read O only after all earlier ones are done.

    The P V issuer of tile t issues P V_t(j) only once the S issuer has issued
    S_t(j+1) (when the item has one), so that P V products never queue ahead of a
    pending S product; the S issuer signals each issue on s_issued{t}{g % 2}.

    Mutations that must be caught: ``s_waits_free=False`` (the S issuer does not
    wait for the S buffer to be copied out), ``p_waits_pv=False`` (the softmax
    stores P_t(g) without waiting for P V_t(g-1), and rescales O without it),
    ``s_issued_barriers=1`` (one s_issued barrier per tile: the S issuer can run
    two phases ahead of the P V issuer's wait)."""
    rnd = random.Random(seed)
    B = {}
    BK128 = 128
    NW = 8

    def bar(name, count):
        B[name] = Bar(name, count)

    for t in range(2):
        for name, c in (("q_full", 1), ("q_empty", 1), ("s_full", 1), ("p_full", BQ), ("pv_done0", 1),
                        ("pv_done1", 1)):
            bar(f"{name}{t}", c)
    bar("s_free", BQ)
    for t in range(2):
        for b in range(2):
            bar(f"s_issued{t}{b}", 1)
    for s_ in range(rk):
        bar(f"k_full{s_}", 1)
        bar(f"k_empty{s_}", 1)
    for s_ in range(rv):
        bar(f"v_full{s_}", 1)
        bar(f"v_empty{s_}", 2)
    consumers = 4 + NW
    for s_ in range(item_ring):
        bar(f"item_full{s_}", 1)
        bar(f"item_empty{s_}", consumers)
    tensor_pipe, tma = [], []
    late = [[], []]          # per tile: P V commits executed but not yet arrived (in order)
    o_done = [-1, -1]        # per tile: the last P V product whose commit has arrived
    o_last = [None, None]    # per tile: the last P V product executed
    sbuf = [None]            # the S buffer: (tile, block index of the tile)
    sreads = {}              # (tile, g) -> softmax warps that copied it out
    pbuf = [[None] * 4 for _ in range(2)]  # per tile and lane quadrant: ("P", g)
    pv_read = [set(), set()]

    def nkv(n_seq, q0, t):
        r0 = q0 + t * BQ
        if r0 >= n_seq:
            return 0
        if not causal:
            return (n_seq + BK128 - 1) // BK128
        return (min(n_seq, r0 + BQ) - 1) // BK128 + 1

    def counts(q0):
        if isinstance(q0, int):
            q0, n_seq, nrow = q0, N, N
        elif len(q0) == 2:
            (q0, n_seq), nrow = q0, q0[1]
        else:
            q0, n_seq, nrow = q0
        n = [nkv(n_seq, q0, t) if q0 + t * BQ < nrow else 0 for t in range(2)]
        return n, max(n)

    def take(i):
        if item_ring:
            yield ("wait", f"item_full{i % item_ring}", i // item_ring)
            yield ("arrive", f"item_empty{i % item_ring}", 1)

    def scheduler():
        for i in range(len(items) + 1):
            yield ("wait", f"item_empty{i % item_ring}", i // item_ring - 1)
            yield ("arrive", f"item_full{i % item_ring}", 1)

    def producer():
        qcount, kpos, vpos = [0, 0], 0, 0
        for i, q0 in enumerate(items):
            yield from take(i)
            n, nmax = counts(q0)
            for t in range(2):
                if n[t]:
                    yield ("wait", f"q_empty{t}", qcount[t] - 1)
                    tma.append(f"q_full{t}")
                    qcount[t] += 1
            order = (["K"] if nmax > 0 else []) + [x for j in range(nmax)
                                                   for x in (["K"] if j + 1 < nmax else []) + ["V"]]
            for kind in order:
                if kind == "K":
                    yield ("wait", f"k_empty{kpos % rk}", kpos // rk - 1)
                    tma.append(f"k_full{kpos % rk}")
                    kpos += 1
                else:
                    yield ("wait", f"v_empty{vpos % rv}", vpos // rv - 1)
                    tma.append(f"v_full{vpos % rv}")
                    vpos += 1
        yield from take(len(items))

    def s_issuer():
        qcount, kpos, issued = [0, 0], 0, 0
        g0 = [0, 0]
        for i, q0 in enumerate(items):
            yield from take(i)
            n, nmax = counts(q0)
            for t in range(2):
                if n[t]:
                    yield ("wait", f"q_full{t}", qcount[t])
                    qcount[t] += 1
            for j in range(nmax):
                s_ = kpos % rk
                yield ("wait", f"k_full{s_}", kpos // rk)
                kpos += 1
                for t in range(2):
                    if j >= n[t]:
                        continue
                    if issued and s_waits_free:
                        yield ("wait", "s_free", issued - 1)
                    issued += 1
                    tensor_pipe.extend([("mma", "S", t, g0[t] + j), ("commit", f"s_full{t}")]
                                       + ([("commit", f"q_empty{t}")] if j == n[t] - 1 else []))
                    gi = g0[t] + j
                    yield ("arrive", f"s_issued{t}{gi % s_issued_barriers}", 1)
                tensor_pipe.append(("commit", f"k_empty{s_}"))
            for t in range(2):
                g0[t] += n[t]
        yield from take(len(items))

    def pv_issuer(t):
        vpos = pcount = 0
        for i, q0 in enumerate(items):
            yield from take(i)
            n, nmax = counts(q0)
            for j in range(nmax):
                s_ = vpos % rv
                yield ("wait", f"v_full{s_}", vpos // rv)
                vpos += 1
                if j >= n[t]:
                    yield ("arrive", f"v_empty{s_}", 1)
                    continue
                yield ("wait", f"p_full{t}", pcount)
                if pv_after_next_s and j + 1 < n[t]:  # S_t of the next block is issued first
                    nxt = pcount + 1
                    yield ("wait", f"s_issued{t}{nxt % s_issued_barriers}", nxt // s_issued_barriers)
                tensor_pipe.extend([("mma", "PV", t, pcount), ("late", t, pcount), ("commit", f"v_empty{s_}")])
                pcount += 1
        yield from take(len(items))

    def softmax(w):
        t, q = w // 4, w % 4
        scount = g = 0
        for i, q0 in enumerate(items):
            yield from take(i)
            n, _ = counts(q0)
            if not n[t]:
                continue
            for j in range(n[t]):
                yield ("wait", f"s_full{t}", scount)
                scount += 1
                assert sbuf[0] == (t, g), f"softmax {w} expects S({t}, {g}) but the buffer holds {sbuf[0]}"
                sreads[(t, g)] = sreads.get((t, g), 0) + 1
                yield ("arrive", "s_free", 32)
                if g > 0 and p_waits_pv:
                    yield ("wait", f"pv_done{t}{(g - 1) & 1}", (g - 1) >> 1)
                cell = pbuf[t][q]
                assert cell is None or cell[1] in pv_read[t], (
                    f"tile {t}: P({g}) overwrites P{cell} before its P V product read it")
                pbuf[t][q] = ("P", g)
                if j > 0 and rnd.random() < rescale_prob:
                    assert o_done[t] >= g - 1, f"tile {t}: O rescaled before P V({g - 1}) is done"
                yield ("arrive", f"p_full{t}", 32)
                g += 1
            yield ("wait", f"pv_done{t}{(g - 1) & 1}", (g - 1) >> 1)  # epilogue
            assert o_done[t] == g - 1, f"tile {t}: the epilogue reads O with P V done up to {o_done[t]}"
            assert o_last[t] == g - 1, f"tile {t}: the epilogue reads O after P V({o_last[t]})"
        yield from take(len(items))

    def execute(kind, t, g):
        if kind == "S":
            prev = sbuf[0]
            assert prev is None or sreads.get(prev, 0) == 4, (
                f"S({t}, {g}) overwrites S{prev} copied out by {sreads.get(prev, 0)} of 4 warps")
            sbuf[0] = (t, g)
        else:
            for cell in pbuf[t]:
                assert cell == ("P", g), f"tile {t}: P V({g}) reads {cell}"
            pv_read[t].add(g)
            o_last[t] = g

    agents = {"producer": producer(), "S": s_issuer(), "PV0": pv_issuer(0), "PV1": pv_issuer(1)}
    if item_ring:
        agents["scheduler"] = scheduler()
    for w in range(NW):
        agents[f"softmax{w}"] = softmax(w)
    waiting = {k: None for k in agents}
    while agents or tensor_pipe or tma or late[0] or late[1]:
        ready = [k for k in agents if waiting[k] is None or B[waiting[k][1]].done(waiting[k][2])]
        if tensor_pipe:
            ready.append("#tensor")
        if tma:
            ready.append("#tma")
        for t in range(2):
            if late[t] and (rnd.random() < late_weight or not ready):
                ready.append(f"#late{t}")
        if not ready:
            raise Deadlock(f"deadlock: {[(k, waiting[k]) for k in agents]}")
        c = rnd.choice(ready)
        if c == "#tensor":
            op = tensor_pipe.pop(0)
            if op[0] == "mma":
                execute(op[1], op[2], op[3])
            elif op[0] == "late":
                late[op[1]].append(op[2])
            else:
                B[op[1]].arrive(1)
            continue
        if c.startswith("#late"):
            t = int(c[-1])
            gdone = late[t].pop(0)
            o_done[t] = gdone
            B[f"pv_done{t}{gdone & 1}"].arrive(1)
            continue
        if c == "#tma":
            B[tma.pop(rnd.randrange(len(tma)))].arrive(1)
            continue
        try:
            while True:
                ev = next(agents[c])
                if ev[0] == "arrive":
                    B[ev[1]].arrive(ev[2])
                    continue
                waiting[c] = ev
                break
        except StopIteration:
            del agents[c]
            waiting[c] = None
    return True


def simulate_bwd_split(n_it, stages, seed, acc_waits=True, qd_empty_count=2, acc_waits_dq_free=True,
                       acc_waits_qd=True):
    """The d = 64 backward with two issuing warps: warp 1 issues every S/dP product, warp 2 the
    dV/dK products of each half and dQ of the block. Each warp's products run in order in their own
    queue; the two queues interleave arbitrarily (they share the tensor core). Besides the barriers,
    the model tracks what each buffer holds, so that these hazards fail here:
      - P^T of half h overwritten by the next pass before dV(i, h) read it (acc_done(h) guards it);
      - a Q/dO stage refilled before both warps' products read it (qd_empty takes two commits);
      - the dQ columns overwritten before both warpgroups read dQ(i) out (dq_free);
      - dS rows (the half's rows of buffer i & 1) overwritten, or used as dQ staging, before dK(i, h)
        and dQ(i) read them;
      - S/dP of a half overwritten before its pass read them.
    Mutations that must be caught: acc_waits=False (no acc_done wait before the P^T store),
    qd_empty_count=1, acc_waits_dq_free=False, acc_waits_qd=False is allowed (the p_full chain
    orders the copies) but modelled to show the stage content is right either way."""
    rnd = random.Random(seed)
    B = {}
    for name, c in (("kv", 1), ("dq_full", 1), ("dq_free", 256), ("drain", 2)):
        B[name] = Bar(name, c)
    for h in range(2):
        for name, c in (("sp_full", 1), ("p_full", 128), ("stats", 128), ("acc_done", 1)):
            B[f"{name}{h}"] = Bar(f"{name}{h}", c)
    for s in range(stages):
        B[f"qd_full{s}"] = Bar(f"qd_full{s}", 1)
        B[f"qd_empty{s}"] = Bar(f"qd_empty{s}", qd_empty_count)
    # buffer contents
    stage = [None] * stages                       # block whose Q/dO a stage holds
    sdp = [None, None]                            # block whose S/dP a half's columns hold
    pt = [[None] * 4 for _ in range(2)]           # block whose packed P^T a half's warp rows hold
    ds = [[[None] * 4 for _ in range(2)] for _ in range(2)]  # [buffer][half][warp] -> ("dS"|"stage", block)
    dq = [None]                                   # block whose dQ the dQ columns hold
    q1, q2, tma = [], [], []

    def s_mma(i, h):
        def run():
            assert stage[i % stages] == i, f"S({i},{h}) reads stage {i % stages} holding {stage[i % stages]}"
            sdp[h] = i
        return ("mma", run)

    def acc_mma(i, h):
        def run():
            assert stage[i % stages] == i, f"acc({i},{h}) reads stage {i % stages} holding {stage[i % stages]}"
            assert all(x == i for x in pt[h]), f"dV({i},{h}) reads P^T {pt[h]}"
            assert all(x == ("dS", i) for x in ds[i & 1][h]), f"dK({i},{h}) reads dS rows {ds[i & 1][h]}"
        return ("mma", run)

    def dq_mma(i):
        def run():
            for h in range(2):
                assert all(x == ("dS", i) for x in ds[i & 1][h]), f"dQ({i}) reads dS rows {ds[i & 1][h]}"
            dq[0] = i
        return ("mma", run)

    def producer():
        tma.append(("kv", None))
        for it in range(n_it):
            s = it % stages
            yield ("wait", f"qd_empty{s}", it // stages - 1)
            tma.append((f"qd_full{s}", (s, it)))

    def warp1():
        yield ("wait", "kv", 0)
        yield ("wait", "qd_full0", 0)
        q1.extend([s_mma(0, 0), ("commit", "sp_full0"), s_mma(0, 1), ("commit", "sp_full1"),
                   ("commit", "qd_empty0")])
        for it in range(n_it):
            nxt = it + 1 < n_it
            yield ("wait", "p_full0", it)
            if nxt:
                s1 = (it + 1) % stages
                yield ("wait", f"qd_full{s1}", (it + 1) // stages)
                q1.extend([s_mma(it + 1, 0), ("commit", "sp_full0")])
            yield ("wait", "p_full1", it)
            if nxt:
                q1.extend([s_mma(it + 1, 1), ("commit", "sp_full1"), ("commit", f"qd_empty{(it + 1) % stages}")])
        q1.append(("commit", "drain"))
        yield ("wait", "drain", 0)

    def warp2():
        for it in range(n_it):
            s = it % stages
            yield ("wait", "p_full0", it)
            if acc_waits_qd:
                yield ("wait", f"qd_full{s}", it // stages)
            q2.extend([acc_mma(it, 0), ("commit", "acc_done0")])
            yield ("wait", "p_full1", it)
            q2.extend([acc_mma(it, 1), ("commit", "acc_done1"), ("commit", f"qd_empty{s}")])
            if it > 0 and acc_waits_dq_free:
                yield ("wait", "dq_free", it - 1)
            q2.extend([dq_mma(it), ("commit", "dq_full")])
        q2.append(("commit", "drain"))

    def grads(h, w):
        def readout(blk):
            yield ("wait", "dq_full", blk)
            assert dq[0] == blk, f"readout({blk}) finds dQ of block {dq[0]}"
            yield ("arrive", "dq_free", 32)
            # stage this warp's dQ rows in its rows of half h of buffer blk & 1 (the bulk reduction has read
            # them before the same warp writes there again)
            assert ds[blk & 1][h][w] == ("dS", blk)
            ds[blk & 1][h][w] = ("stage", blk)
        for it in range(n_it):
            yield ("arrive", f"stats{h}", 32)
            yield ("wait", f"stats{h}", it)
            yield ("wait", f"sp_full{h}", it)
            assert sdp[h] == it, f"pass({it},{h}) reads S/dP of block {sdp[h]}"
            if it > 0 and acc_waits:
                yield ("wait", f"acc_done{h}", it - 1)
            pt[h][w] = it
            ds[it & 1][h][w] = ("dS", it)
            yield ("arrive", f"p_full{h}", 32)
            # S/dP of this half may be overwritten from here on
            if it > 0:
                yield from readout(it - 1)
        yield from readout(n_it - 1)

    agents = {"producer": producer(), "warp1": warp1(), "warp2": warp2()}
    for h in range(2):
        for w in range(4):
            agents[f"g{h}.{w}"] = grads(h, w)
    waiting = {k: None for k in agents}
    while agents or q1 or q2 or tma:
        ready = [k for k in agents if waiting[k] is None or B[waiting[k][1]].done(waiting[k][2])]
        if q1:
            ready.append("#q1")
        if q2:
            ready.append("#q2")
        if tma:
            ready.append("#tma")
        if not ready:
            raise Deadlock(f"deadlock: {[(k, waiting[k]) for k in agents]}")
        c = rnd.choice(ready)
        if c in ("#q1", "#q2"):
            q = q1 if c == "#q1" else q2
            kind, x = q.pop(0)
            if kind == "mma":
                x()
            else:
                B[x].arrive(1)
            continue
        if c == "#tma":
            name, load = tma.pop(rnd.randrange(len(tma)))
            if load is not None:
                stage[load[0]] = load[1]
            B[name].arrive(1)
            continue
        try:
            while True:
                ev = next(agents[c])
                if ev[0] == "arrive":
                    B[ev[1]].arrive(ev[2])
                    continue
                waiting[c] = ev
                break
        except StopIteration:
            del agents[c]
            waiting[c] = None
    return True


def simulate_bwd128_split(n_it, stages, seed, sp_count=2, dq_count=2, q_empty_count=2, waits_dq_free=True,
                          do_empty_count=8, release_after_read=True):
    """The d = 128 backward with two issuing warps: warp 1 issues S^T, dV and dQ's first 64 head
    columns, warp 2 dP^T, dK and dQ's second half; each warp's products run in order in their own
    queue. The tensor-memory columns alias (S^T, then packed P^T and dQ half 0 in [0, 128); dP^T,
    then dS^T and dQ half 1 in [128, 256)), so the model tracks which block each holds: a product
    that overwrites columns before their last reader, or a reader that finds the wrong block,
    fails. Completion barriers count a commit from each warp (sp_full, dq_full, q_empty, drain).
    A stage's Q and dO halves have their own barriers: Q goes back to the producer by the issuing
    warps' commits, dO by the eight gradient warps, because each stages its second dQ tile there
    (its first in its own dS rows) and releases it once its bulk reductions have read it, which it
    waits for at its next pass. The model keeps those reads pending until that wait, so a dO copy
    landing on a tile not yet read fails.
    Mutations that must be caught: sp_count=1, dq_count=1, q_empty_count=1, waits_dq_free=False,
    do_empty_count=7, release_after_read=False (released when staged)."""
    rnd = random.Random(seed)
    B = {}
    n = 256
    for name, c in (("kv", 1), ("sp_full", sp_count), ("p_full", n), ("dq_full", dq_count), ("dq_free", n),
                    ("drain", 2), ("stats", n)):
        B[name] = Bar(name, c)
    for s in range(stages):
        B[f"q_full{s}"] = Bar(f"q_full{s}", 1)
        B[f"q_empty{s}"] = Bar(f"q_empty{s}", q_empty_count)
        B[f"do_full{s}"] = Bar(f"do_full{s}", 1)
        B[f"do_empty{s}"] = Bar(f"do_empty{s}", do_empty_count)
    stage_q, stage_do = [None] * stages, [None] * stages
    do_tiles = [set() for _ in range(stages)]  # warps whose dQ tile in a stage's dO half is not read yet
    # per half of the tensor memory (0: S^T side, 1: dP^T side): what the columns hold
    cols = [{"sdp": None, "packed": None, "dq": None} for _ in range(2)]
    packed_read = [None, None]   # last block whose packed P^T / dS^T the dV / dK product read
    dq_read = [set(), set()]      # (block, warp) pairs that read dQ half h out
    ds_smem = [None]              # ("dS" | "stage", block) of the shared-memory dS buffer
    qs = [[], []]
    tma = []

    def prod(h, kind, i):
        def run():
            s = i % stages
            assert stage_q[s] == i and stage_do[s] == i, f"{kind}({i}) reads stage {s}: Q {stage_q[s]}, dO {stage_do[s]}"
            c = cols[h]
            if kind == "sdp":
                if i > 0:
                    assert packed_read[h] == i - 1, f"S/dP({i}) over packed columns dV/dK({i - 1}) did not read"
                    assert all((i - 1, w) in dq_read[h] for w in range(8)), f"S/dP({i}) over dQ({i - 1}) half {h}"
                c["sdp"] = i
            elif kind == "acc":
                assert c["packed"] == i, f"dV/dK({i}) half {h} reads packed block {c['packed']}"
                packed_read[h] = i
            else:  # dq
                assert ds_smem[0] == ("dS", i), f"dQ({i}) reads dS {ds_smem[0]}"
                c["dq"] = i
        return ("mma", run)

    def producer():
        tma.append(("kv", None))
        for it in range(n_it):
            s = it % stages
            yield ("wait", f"q_empty{s}", it // stages - 1)
            tma.append((f"q_full{s}", ("q", s, it)))
            yield ("wait", f"do_empty{s}", it // stages - 1)
            tma.append((f"do_full{s}", ("do", s, it)))

    def issuer(h):
        yield ("wait", "kv", 0)
        for it in range(n_it):
            s = it % stages
            yield ("wait", f"q_full{s}", it // stages)
            yield ("wait", f"do_full{s}", it // stages)
            if it > 0 and waits_dq_free:
                yield ("wait", "dq_free", it - 1)
            qs[h].extend([prod(h, "sdp", it), ("commit", "sp_full")])
            yield ("wait", "p_full", it)
            qs[h].extend([prod(h, "acc", it), prod(h, "dq", it), ("commit", "dq_full"), ("commit", f"q_empty{s}")])
        qs[h].append(("commit", "drain"))
        if h == 0:
            yield ("wait", "drain", 0)

    def grads(w):
        for it in range(n_it):
            yield ("arrive", "stats", 32)
            yield ("wait", "stats", it)
            yield ("wait", "sp_full", it)
            assert cols[0]["sdp"] == it and cols[1]["sdp"] == it, f"pass({it}) finds S/dP {cols[0]['sdp']}, {cols[1]['sdp']}"
            cols[0]["packed"] = cols[1]["packed"] = it
            # before its first dS store (its own rows) the warp waits for its last block's reductions to have
            # read both of its tiles; then the dO half of that block's stage can go back to the producer
            if it > 0:
                sp = (it - 1) % stages
                do_tiles[sp].discard(w)
                if release_after_read:
                    yield ("arrive", f"do_empty{sp}", 1)
            ds_smem[0] = ("dS", it)
            yield ("arrive", "p_full", 32)
            yield ("wait", "dq_full", it)
            assert cols[0]["dq"] == it and cols[1]["dq"] == it, f"readout({it}) finds dQ {cols[0]['dq']}, {cols[1]['dq']}"
            dq_read[0].add((it, w))
            dq_read[1].add((it, w))
            yield ("arrive", "dq_free", 32)
            ds_smem[0] = ("stage", it)
            s = it % stages
            assert stage_do[s] == it, f"readout({it}) stages into a dO half holding block {stage_do[s]}"
            do_tiles[s].add(w)  # pending until this warp's wait at its next pass
            if not release_after_read:
                yield ("arrive", f"do_empty{s}", 1)

    agents = {"producer": producer(), "w1": issuer(0), "w2": issuer(1)}
    for w in range(8):
        agents[f"g{w}"] = grads(w)
    waiting = {k: None for k in agents}
    while agents or qs[0] or qs[1] or tma:
        ready = [k for k in agents if waiting[k] is None or B[waiting[k][1]].done(waiting[k][2])]
        for h in range(2):
            if qs[h]:
                ready.append(f"#q{h}")
        if tma:
            ready.append("#tma")
        if not ready:
            raise Deadlock(f"deadlock: {[(k, waiting[k]) for k in agents]}")
        c = rnd.choice(ready)
        if c.startswith("#q"):
            kind, x = qs[int(c[2])].pop(0)
            if kind == "mma":
                x()
            else:
                B[x].arrive(1)
            continue
        if c == "#tma":
            name, load = tma.pop(rnd.randrange(len(tma)))
            if load is not None:
                kind, st, blk = load
                if kind == "q":
                    stage_q[st] = blk
                else:
                    assert not do_tiles[st], f"dO({blk}) lands on dQ tiles of warps {do_tiles[st]} not yet read"
                    stage_do[st] = blk
            B[name].arrive(1)
            continue
        try:
            while True:
                ev = next(agents[c])
                if ev[0] == "arrive":
                    B[ev[1]].arrive(ev[2])
                    continue
                waiting[c] = ev
                break
        except StopIteration:
            del agents[c]
            waiting[c] = None
    return True
