"""A randomised model of the mbarrier protocols of the tensor-core kernels.

Each role of a kernel (the TMA warp, the MMA warp, several elementwise or
softmax warps) is a Python generator that yields the barrier operations of the
kernel's code, in the kernel's order:

  ("wait", bar, k)   wait for completion k (0-based) of `bar`, as
                     mbar_wait(bar, k & 1) does: a parity wait returns once
                     the completion count is odd/even, not once it exceeds k
  ("arrive", bar)    one arrival (a warp stands for all of its threads)
  ("mma", label)     an MMA issued to the tensor pipe (no barrier effect)
  ("commit", bar)    tcgen05.commit: an arrival on `bar` once every MMA issued
                     before it has completed
  ("tma", bar)       a TMA copy whose completion arrives on `bar`

Two asynchronous agents run beside the roles: the tensor pipe, which runs the
MMA warp's products and commits in issue order, and the TMA engine, whose
copies complete in any order.  A seeded scheduler picks one runnable agent at
random at every step.

Checked on every step of every schedule:
  1. no role waits for completion k of a barrier that has completed k + 2 or
     more times (its parity wait would miss the phase it waits for);
  2. every arrival lands in the phase it belongs to: the arrival of a role
     for its m-th use of a barrier is counted while the barrier is in phase m
     (an arrival that overtakes would complete an earlier phase early);
  3. no deadlock: while some role has not finished, some agent can run.

The kernels' protocols are written out below, one function per kernel, from
their sources (tc_fwd.cu, tc_bwd2.cu); `Item` lists describe the work that
the persistent CTA receives.  Only barriers are modelled: tensor-memory and
shared-memory contents are not.
"""
import random
from collections import defaultdict


class ProtocolError(Exception):
    pass


class _Bar:
    __slots__ = ("need", "done", "pending")

    def __init__(self, need):
        self.need = need
        self.done = 0
        self.pending = 0


class Sim:
    """One schedule of one CTA.  `need` maps barrier name -> arrivals per phase."""

    def __init__(self, need, seed, skip_waits=()):
        self.need = need
        self.skip_waits = frozenset(skip_waits)  # planted mistakes: waits left out
        self.rnd = random.Random(seed)
        self.bars = {}
        self.uses = defaultdict(int)  # (agent, bar) -> arrivals so far
        self.pipe = []  # tensor pipe FIFO: ("mma", label) or ("commit", bar)
        self.copies = []  # TMA copies in flight: bar names

    def bar(self, name):
        b = self.bars.get(name)
        if b is None:
            b = self.bars[name] = _Bar(self.need[name])
        return b

    def arrive(self, who, name):
        b = self.bar(name)
        m = self.uses[(who, name)]
        self.uses[(who, name)] = m + 1
        if m != b.done:
            raise ProtocolError(
                f"{who}: arrival for phase {m} of {name} counted in phase {b.done}")
        b.pending += 1
        if b.pending == b.need:
            b.pending = 0
            b.done += 1

    def run(self, roles, max_steps=10 ** 6):
        """Run `roles` (name -> generator) to the end; raises ProtocolError."""
        blocked = {}
        live = dict(roles)
        for name, g in list(live.items()):
            try:
                blocked[name] = next(g)
            except StopIteration:
                del live[name]
        steps = 0
        while live or self.pipe or self.copies:
            steps += 1
            if steps > max_steps:
                raise ProtocolError("step limit")
            ready = []
            for name in live:
                op = blocked[name]
                if op[0] == "wait" and op[1] in self.skip_waits:
                    ready.append(name)
                elif op[0] == "wait":
                    _, bname, k = op
                    b = self.bar(bname)
                    if b.done >= k + 2:
                        raise ProtocolError(
                            f"{name} waits for completion {k} of {bname}, which has "
                            f"completed {b.done} times (a parity wait misses it)")
                    if b.done == k + 1:
                        ready.append(name)
                else:
                    ready.append(name)
            if self.pipe:
                ready.append("@pipe")
            if self.copies:
                ready.append("@tma")
            if not ready:
                raise ProtocolError(f"deadlock: {blocked}")
            who = self.rnd.choice(ready)
            if who == "@pipe":
                op = self.pipe.pop(0)
                if op[0] == "commit":
                    self.arrive("@pipe", op[1])
                continue
            if who == "@tma":
                bname = self.copies.pop(self.rnd.randrange(len(self.copies)))
                self.arrive("@tma", bname)
                continue
            op = blocked[who]
            kind = op[0]
            if kind == "arrive":
                self.arrive(who, op[1])
            elif kind in ("mma", "commit"):
                self.pipe.append(op)
            elif kind == "tma":
                self.copies.append(op[1])
            elif kind != "wait":
                raise ProtocolError(f"unknown op {op}")
            try:
                blocked[who] = live[who].send(None)
            except StopIteration:
                del live[who]
                del blocked[who]


def _take_item(ring, nitem):
    """Consumer side of the two-entry item ring (all three kernels)."""
    e = nitem & 1
    yield ("wait", f"ITEMF{e}", nitem >> 1)
    t = ring[e]
    yield ("arrive", f"ITEME{e}")
    return t


def _give_items(ring, n_items):
    """Producer side of the ring, as the TMA warp runs it (one step per item)."""
    for nitem in range(n_items + 1):
        e = nitem & 1
        if nitem >= 2:
            yield ("wait", f"ITEME{e}", (nitem >> 1) - 1)
        ring[e] = nitem if nitem < n_items else -1
        yield ("arrive", f"ITEMF{e}")
        if nitem == n_items:
            return
        yield nitem


def _ring_fill(slot_bar_empty, slot_bar_full, fill):
    """TMA fill number `fill` of a ring slot: wait for the previous fill's release."""
    if fill >= 1:
        yield ("wait", slot_bar_empty, fill - 1)
    yield ("tma", slot_bar_full)


# ---------------------------------------------------------------------------
# Query-major reverse kernel (tc_bwd_q_kernel): items are query blocks, each
# with a number of non-empty key blocks.
# ---------------------------------------------------------------------------
def dq_kernel(blocks, ew_warps=3, two_ds=True, NK=3, NV=1):
    """Roles of the dQ kernel (tc_bwd_q_kernel) for items with blocks[n] key
    blocks each: TMA, MMA and the elementwise warps, which also form delta
    (meeting at B_DPART) and run the dQ epilogue (B_DONE / B_DREAD, staging
    tile: B_EPIF / B_EPI).

    two_ds=False models its first form, with one dS barrier (waited with
    parity t & 1), which a schedule can break: the elementwise warps complete
    dS(t) and dS(t + 1) before the MMA warp's first poll of dS(t)."""
    W = ew_warps
    need = defaultdict(lambda: 1)
    for e in (0, 1):
        need[f"ITEME{e}"] = 1 + W
    for b in ("DS0", "DS1", "SFREE", "DREAD", "EPI", "DPART"):
        need[b] = W
    ring = [None, None]
    N = len(blocks)

    def ds_bar(t):
        return (f"DS{t & 1}", t >> 1) if two_ds else ("DS0", t)

    def tma():
        it = 0
        gen = _give_items(ring, N)
        for op in gen:
            if isinstance(op, tuple):
                yield op
                continue
            nitem = op
            if nitem > 0:
                yield ("wait", "QFREE", nitem - 1)
            yield ("tma", "Q")
            for _ in range(blocks[nitem]):
                yield from _ring_fill(f"KVE{NK + it % NV}", f"KVF{NK + it % NV}", it // NV)
                yield from _ring_fill(f"KVE{it % NK}", f"KVF{it % NK}", it // NK)
                it += 1
        for u in range(min(NK, it)):
            i = it - 1 - u
            yield ("wait", f"KVF{i % NK}", i // NK)
        for u in range(min(NV, it)):
            i = it - 1 - u
            yield ("wait", f"KVF{NK + i % NV}", i // NV)
        if N > 0:
            yield ("wait", "Q", N - 1)

    def mma():
        t = ne = 0
        for nitem in range(N + 1):
            ti = yield from _take_item(ring, nitem)
            if ti < 0:
                break
            k = blocks[ti]
            yield ("wait", "Q", nitem)
            t0 = t

            def free_q():
                if k > 0:
                    yield ("wait", "DPART", ne)
                yield ("commit", "QFREE")

            def issue_dp(tt):
                yield ("wait", f"KVF{NK + tt % NV}", tt // NV)
                yield ("mma", f"dP{tt}")
                yield ("commit", f"KVE{NK + tt % NV}")

            def issue_s(tt):
                yield ("wait", f"KVF{tt % NK}", tt // NK)
                yield ("mma", f"S{tt}")
                yield ("commit", "SDP")

            if k > 0:
                yield from issue_dp(t)
                if t > 0:
                    yield ("wait", "SFREE", t - 1)
                yield from issue_s(t)
            if k <= 1:
                yield from free_q()
            for b in range(k):
                if b + 1 < k:
                    yield from issue_dp(t + 1)
                    yield ("wait", "SFREE", t)
                    yield from issue_s(t + 1)
                    if b + 2 >= k:
                        yield from free_q()
                bname, kk = ds_bar(t)
                yield ("wait", bname, kk)
                yield ("mma", f"dQ{t}")
                yield ("commit", f"KVE{t % NK}")
                t += 1
            assert t - t0 == k
            if k > 0:
                ne += 1
            if nitem > 0:
                yield ("wait", "DREAD", nitem - 1)
            yield ("commit", "DONE")
        yield ("commit", "DRAIN")
        yield ("wait", "DRAIN", 0)

    def ew(w):
        t = ne = 0
        ti = yield from _take_item(ring, 0)
        nitem = 0
        while ti >= 0:
            k = blocks[ti]
            if k > 0:
                yield ("wait", "Q", nitem)
                # delta reads this item's dY from shared memory up to its DPART
                # arrival: the next item's Q, dY load must not have landed yet
                # (a second completion of Q ahead shows as a missed parity).
                yield ("wait", "Q", nitem)
                yield ("arrive", "DPART")
                yield ("wait", "DPART", ne)
                ne += 1
            for _ in range(k):
                yield ("wait", "SDP", t)
                yield ("arrive", "SFREE")
                yield ("arrive", ds_bar(t)[0])
                t += 1
            tn = yield from _take_item(ring, nitem + 1)
            yield ("wait", "DONE", nitem)
            yield ("arrive", "DREAD")
            if w == 0:
                yield ("arrive", "EPIF")
            yield ("wait", "EPIF", nitem)
            yield ("arrive", "EPI")
            if w == 0:
                yield ("wait", "EPI", nitem)
            ti = tn
            nitem += 1

    roles = {"tma": tma(), "mma": mma()}
    for w in range(W):
        roles[f"ew{w}"] = ew(w)
    return need, roles


# ---------------------------------------------------------------------------
# Key-major reverse kernel (tc_bwd_kv_kernel): items are key blocks, each with
# a number of non-empty query blocks.
# ---------------------------------------------------------------------------
def kv_kernel(blocks, ew_warps=4, NST=2):
    W = ew_warps
    assert W % 2 == 0
    need = defaultdict(lambda: 1)
    for e in (0, 1):
        need[f"ITEME{e}"] = 1 + W
    for b in ("P", "DSB", "ACCFREE"):
        need[b] = W
    need["EPIV"] = need["EPIK"] = W // 2
    ring = [None, None]
    N = len(blocks)

    def tma():
        it = 0
        for op in _give_items(ring, N):
            if isinstance(op, tuple):
                yield op
                continue
            nitem = op
            if nitem > 0:
                yield ("wait", "KVFREE", nitem - 1)
            yield ("tma", "KV")
            for _ in range(blocks[nitem]):
                yield from _ring_fill(f"QE{it % NST}", f"QF{it % NST}", it // NST)
                it += 1
        for u in range(min(NST, it)):
            i = it - 1 - u
            yield ("wait", f"QF{i % NST}", i // NST)
        if N > 0:
            yield ("wait", "KV", N - 1)

    def mma():
        it = 0
        for nitem in range(N + 1):
            ti = yield from _take_item(ring, nitem)
            if ti < 0:
                break
            k = blocks[ti]
            yield ("wait", "KV", nitem)
            it0 = it
            if k > 0:
                yield ("wait", f"QF{it % NST}", it // NST)
                yield ("mma", f"S{it}")
                yield ("commit", "S")
                yield ("mma", f"dP{it}")
                yield ("commit", "DP")
            if k <= 1:
                yield ("commit", "KVFREE")
            for b in range(k):
                slot = it % NST
                more = b + 1 < k
                yield ("wait", "P", it)
                if it == it0 and nitem > 0:
                    yield ("wait", "ACCFREE", nitem - 1)
                yield ("mma", f"dV{it}")
                if more:
                    yield ("wait", f"QF{(it + 1) % NST}", (it + 1) // NST)
                    yield ("mma", f"S{it + 1}")
                    yield ("commit", "S")
                yield ("wait", "DSB", it)
                yield ("mma", f"dK{it}")
                yield ("commit", f"QE{slot}")
                if more:
                    yield ("mma", f"dP{it + 1}")
                    yield ("commit", "DP")
                    if b + 2 >= k:
                        yield ("commit", "KVFREE")
                it += 1
            if it == it0 and nitem > 0:
                yield ("wait", "ACCFREE", nitem - 1)
            yield ("commit", "DONE")
        yield ("commit", "DRAIN")
        yield ("wait", "DRAIN", 0)

    def ew(w):
        is_dv = w < W // 2
        it = 0
        for nitem in range(N + 1):
            ti = yield from _take_item(ring, nitem)
            if ti < 0:
                break
            for _ in range(blocks[ti]):
                yield ("wait", "S", it)
                yield ("arrive", "P")
                yield ("wait", "DP", it)
                yield ("arrive", "DSB")
                it += 1
            yield ("wait", "DONE", nitem)
            yield ("arrive", "ACCFREE")
            if w == W // 2:  # the warp of the dK stores' issuer
                yield ("arrive", "EPIFV")
            yield ("wait", "EPIFV" if is_dv else "EPIFK", nitem)
            yield ("arrive", "EPIV" if is_dv else "EPIK")
            if w in (0, W // 2):  # the issuers of the dV and dK stores
                yield ("wait", "EPIV" if is_dv else "EPIK", nitem)
                if is_dv:
                    yield ("arrive", "EPIFK")

    roles = {"tma": tma(), "mma": mma()}
    for w in range(W):
        roles[f"ew{w}"] = ew(w)
    return need, roles


# ---------------------------------------------------------------------------
# Forward kernel (tc_fwd_kernel): items are pairs of query tiles A, B; each
# has a list of key blocks given as (A non-empty, B non-empty), never both
# empty (blocks empty for both tiles are skipped by every role).
# ---------------------------------------------------------------------------
def fwd_kernel(items, warps_per_tile=2, NS=3):
    W = warps_per_tile
    need = defaultdict(lambda: 1)
    for e in (0, 1):
        need[f"ITEME{e}"] = 1 + 2 * W
    for X in (0, 1):
        need[f"P{X}"] = need[f"OREAD{X}"] = need[f"Y{X}"] = W
    ring = [None, None]
    N = len(items)

    def tma():
        it = 0
        for op in _give_items(ring, N):
            if isinstance(op, tuple):
                yield op
                continue
            nitem = op
            if nitem > 0:
                yield ("wait", "QFREE", nitem - 1)
            yield ("tma", "Q")
            for _ in items[nitem]:
                for _kv in range(2):
                    yield from _ring_fill(f"KVE{it % NS}", f"KVF{it % NS}", it // NS)
                    it += 1
        for u in range(min(NS, it)):
            i = it - 1 - u
            yield ("wait", f"KVF{i % NS}", i // NS)
        if N > 0:
            yield ("wait", "Q", N - 1)

    def mma():
        it = 0
        cnt = [0, 0]
        for nitem in range(N + 1):
            ti = yield from _take_item(ring, nitem)
            if ti < 0:
                break
            blocks = items[ti]
            yield ("wait", "Q", nitem)
            pend_b = have_prev = False
            pend_b_phase = pend_vslot = 0
            if not blocks:
                yield ("commit", "QFREE")
            for bi, (c0, c1) in enumerate(blocks):
                kslot, kph = it % NS, it // NS
                it += 1
                vslot, vph = it % NS, it // NS
                it += 1
                yield ("wait", f"KVF{kslot}", kph)
                if c0:
                    yield ("mma", "S_A")
                    yield ("commit", "S0")
                if pend_b:
                    yield ("wait", "P1", pend_b_phase)
                    yield ("mma", "PV_B")
                if have_prev:
                    yield ("commit", f"KVE{pend_vslot}")
                if c1:
                    yield ("mma", "S_B")
                    yield ("commit", "S1")
                if bi == len(blocks) - 1:
                    yield ("commit", "QFREE")
                yield ("commit", f"KVE{kslot}")
                yield ("wait", f"KVF{vslot}", vph)
                if c0:
                    yield ("wait", "P0", cnt[0])
                    yield ("mma", "PV_A")
                    cnt[0] += 1
                pend_b = c1
                pend_b_phase = cnt[1]
                if pend_b:
                    cnt[1] += 1
                pend_vslot = vslot
                have_prev = True
            if pend_b:
                yield ("wait", "P1", pend_b_phase)
                yield ("mma", "PV_B")
            if have_prev:
                yield ("commit", f"KVE{pend_vslot}")
            for X in (0, 1):
                if nitem > 0:
                    yield ("wait", f"OREAD{X}", nitem - 1)
                yield ("commit", f"O{X}")
        yield ("commit", "DRAIN")
        yield ("wait", "DRAIN", 0)

    def softmax(X, w):
        cnt = 0
        for nitem in range(N + 1):
            ti = yield from _take_item(ring, nitem)
            if ti < 0:
                break
            for blk in items[ti]:
                if not blk[X]:
                    continue
                yield ("wait", f"S{X}", cnt)
                yield ("arrive", f"P{X}")
                cnt += 1
            yield ("wait", f"O{X}", nitem)
            yield ("arrive", f"OREAD{X}")
            if w == 0:  # the issuer of tile X's stores
                yield ("arrive", f"YF{X}")
            yield ("wait", f"YF{X}", nitem)
            yield ("arrive", f"Y{X}")
            if w == 0:
                yield ("wait", f"Y{X}", nitem)

    roles = {"tma": tma(), "mma": mma()}
    for X in (0, 1):
        for w in range(W):
            roles[f"sm{X}.{w}"] = softmax(X, w)
    return need, roles


def run_kernel(factory, work, seed, skip_waits=(), **kw):
    """One random schedule; returns None, or the ProtocolError's text."""
    need, roles = factory(work, **kw)
    try:
        Sim(need, seed, skip_waits).run(roles)
    except ProtocolError as e:
        return str(e)
    return None


def random_counts(rnd, n_items, choices=(0, 1, 1, 2, 3, 5)):
    return [rnd.choice(choices) for _ in range(n_items)]


def random_fwd_items(rnd, n_items):
    items = []
    for _ in range(n_items):
        b_valid = rnd.random() < 0.8
        blocks = []
        for _ in range(rnd.choice((0, 1, 2, 3, 4))):
            a = rnd.random() < 0.85
            b = b_valid and rnd.random() < 0.85
            if not (a or b):
                a = True
            blocks.append((a, b))
        items.append(blocks)
    return items


# ---------------------------------------------------------------------------
# Atomic-dQ reverse kernel (tc_bwd_kernel): one key block per CTA, a number of
# non-empty query blocks; dQ leaves through drain warps.
# ---------------------------------------------------------------------------
def atomic_kernel(n_blocks, ew_warps=2, drain_warps=2):
    W, Dw = ew_warps, drain_warps
    need = defaultdict(lambda: 1)
    need["DS"] = W
    need["DQD"] = Dw
    k = n_blocks

    def tma():
        yield ("tma", "KV")
        for it in range(k):
            yield from _ring_fill(f"QE{it & 1}", f"QF{it & 1}", it >> 1)
        for s in range(min(2, k)):
            i = k - 1 - s
            yield ("wait", f"QF{i & 1}", i >> 1)
        yield ("wait", "KV", 0)

    def mma():
        yield ("wait", "KV", 0)
        for it in range(k):
            yield ("wait", f"QF{it & 1}", it >> 1)
            yield ("mma", "dP")
            if it > 0:
                yield ("wait", "DQD", it - 1)
            yield ("mma", "S")
            yield ("commit", "SDP")
            yield ("wait", "DS", it)
            yield ("mma", "dV")
            yield ("mma", "dK")
            yield ("commit", f"QE{it & 1}")
            yield ("mma", "dQ")
            yield ("commit", "DQF")
        yield ("commit", "DONE")
        yield ("commit", "DRAIN")
        yield ("wait", "DRAIN", 0)

    def ew():
        for it in range(k):
            yield ("wait", "SDP", it)
            yield ("arrive", "DS")
        if k > 0:
            yield ("wait", "DONE", 0)

    def drain():
        for it in range(k):
            yield ("wait", "DQF", it)
            yield ("arrive", "DQD")

    roles = {"tma": tma(), "mma": mma()}
    for w in range(W):
        roles[f"ew{w}"] = ew()
    for w in range(Dw):
        roles[f"drain{w}"] = drain()
    return need, roles


# ---------------------------------------------------------------------------
# 3xTF32 reverse pass (tc_bwd32.cu): one CTA per block, steps of 32 rows.
# ---------------------------------------------------------------------------
def kv32_kernel(n_steps, ew_warps=2, NSS=3, NTS=2, NV=4, promote=3):
    """dK/dV kernel: the elementwise warps write K, V (B_A); the TMA warp fills
    S halves (QSF / QSE) and vector slots (VF / VE) one step ahead of T halves
    (QTF / QTE); S^T, dP^T double-buffered (SP per buffer); P^T and dS^T per
    buffer (P, DS); S^T(t+1), dP^T(t+1) before dV(t), dK(t); every `promote`
    steps the elementwise warps wait for the segment's dV, dK (SEG) before
    moving them out (the kernel's interval is 32: a short one here so that
    SEG turns over within a few steps)."""
    W = ew_warps
    need = defaultdict(lambda: 1)
    for name in ["A", "P0", "P1", "DS0", "DS1"] + [f"VE{s}" for s in range(NV)]:
        need[name] = W
    k = n_steps

    def tma():
        def load_s(s):
            yield from _ring_fill(f"QSE{s % NSS}", f"QSF{s % NSS}", s // NSS)
            yield from _ring_fill(f"VE{s % NV}", f"VF{s % NV}", s // NV)
        if k > 0:
            yield from load_s(0)
        for it in range(k):
            if it + 1 < k:
                yield from load_s(it + 1)
            yield from _ring_fill(f"QTE{it % NTS}", f"QTF{it % NTS}", it // NTS)
        for full, m in (("QSF", NSS), ("QTF", NTS), ("VF", NV)):
            for u in range(min(m, k)):
                i = k - 1 - u
                yield ("wait", f"{full}{i % m}", i // m)

    def mma():
        yield ("wait", "A", 0)
        if k > 0:
            yield ("wait", "QSF0", 0)
            yield ("mma", "SdP0")
            yield ("commit", "SP0")
            yield ("commit", "QSE0")
        for it in range(k):
            b = it & 1
            if it + 1 < k:
                s1 = (it + 1) % NSS
                yield ("wait", f"QSF{s1}", (it + 1) // NSS)
                yield ("mma", f"SdP{it + 1}")
                yield ("commit", f"SP{(it + 1) & 1}")
                yield ("commit", f"QSE{s1}")
            yield ("wait", f"QTF{it % NTS}", it // NTS)
            yield ("wait", f"P{b}", it >> 1)
            yield ("mma", f"dV{it}")
            yield ("wait", f"DS{b}", it >> 1)
            yield ("mma", f"dK{it}")
            if (it + 1) % promote == 0 and it + 1 < k:
                yield ("commit", "SEG")
            yield ("commit", f"QTE{it % NTS}")
        yield ("commit", "DONE")
        yield ("commit", "DRAIN")
        yield ("wait", "DRAIN", 0)

    def ew():
        yield ("arrive", "A")
        for it in range(k):
            b, vs = it & 1, it % NV
            yield ("wait", f"VF{vs}", it // NV)
            yield ("wait", f"SP{b}", it >> 1)
            if it > 0 and it % promote == 0:
                yield ("wait", "SEG", it // promote - 1)
            yield ("arrive", f"VE{vs}")
            yield ("arrive", f"P{b}")
            yield ("arrive", f"DS{b}")
        if k > 0:
            yield ("wait", "DONE", 0)

    roles = {"tma": tma(), "mma": mma()}
    for w in range(W):
        roles[f"ew{w}"] = ew()
    return need, roles


def q32_kernel(n_steps, ew_warps=2, NST=4):
    """dQ kernel: S and dP double-buffered (B_SP per buffer); dS per buffer
    (B_DS); dQ(t) after dS(t), S(t+1) and dP(t+1) before it."""
    W = ew_warps
    need = defaultdict(lambda: 1)
    need["A"] = need["DS0"] = need["DS1"] = W
    k = n_steps

    def tma():
        for it in range(k):
            yield from _ring_fill(f"KE{it % NST}", f"KF{it % NST}", it // NST)
        for u in range(min(NST, k)):
            i = k - 1 - u
            yield ("wait", f"KF{i % NST}", i // NST)

    def mma():
        yield ("wait", "A", 0)
        if k > 0:
            yield ("wait", "KF0", 0)
            yield ("mma", "SdP0")
            yield ("commit", "SP0")
        for t in range(k):
            if t + 1 < k:
                yield ("wait", f"KF{(t + 1) % NST}", (t + 1) // NST)
                yield ("mma", f"SdP{t + 1}")
                yield ("commit", f"SP{(t + 1) & 1}")
            yield ("wait", f"DS{t & 1}", t >> 1)
            yield ("mma", f"dQ{t}")
            yield ("commit", f"KE{t % NST}")
        yield ("commit", "DONE")
        yield ("commit", "DRAIN")
        yield ("wait", "DRAIN", 0)

    def ew():
        yield ("arrive", "A")
        for t in range(k):
            yield ("wait", f"SP{t & 1}", t >> 1)
            yield ("arrive", f"DS{t & 1}")
        if k > 0:
            yield ("wait", "DONE", 0)

    roles = {"tma": tma(), "mma": mma()}
    for w in range(W):
        roles[f"ew{w}"] = ew()
    return need, roles
