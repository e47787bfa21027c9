"""Host models of the attention kernels' barrier protocols, run under random schedules.

The kernel's roles (TMA producer, MMA issuer, compute warps) synchronise through
mbarriers whose waits test a phase *parity*: a wait for phase k returns once
phase k has completed, but if the barrier has meanwhile completed phase k + 1
as well, the parity matches the incomplete phase k + 2 and the waiter hangs
(the kernel's bounded wait then reports a timeout).  The order of products and
barriers must therefore never let a barrier run two phases ahead of one of its
waiters.  At d = 64 the kernel keeps two score buffers and issues the next
step's score product before the current step's P is consumed; each buffer has
its own "scores ready" and "P ready" barrier for that reason.

`Model` replays the protocol of csrc/fa_bwd.cu (the dK/dV kernel; the dQ
kernel's is the same with B = P K in place of dV and dQ~ in place of dK) and
`FwdModel` that of csrc/fa_fwd.cu and `DecodeModel` that of the decode kernel
(csrc/fa_decode.cu), all with true parity semantics: the
tensor core completes products in issue order, a commit's arrival fires when
the products issued before it have completed, tile loads land in any order,
and every role advances at random.  The compute side is two warps that each
own half of every score and dP buffer, arrive on the counting barriers on
their own and may drift a step apart.  It checks over many schedules,
persistent items included, that every run ends (no wait hangs), that every
product and every warp reads the data its step needs (the scores, P and dS of
its own step, not of another), and that no product overwrites data a later
reader still needs.  The forward's issuer sends each key tile's products in
two bursts and tests (without blocking) whether the second group's P is ready
before it commits the first group's scores; its model takes both branches of
that test, and checks the item ring the TMA warp publishes claimed items in.
"""
import random

import pytest


class Barrier:
    def __init__(self, count):
        self.count = count
        self.pending = 0
        self.phases = 0  # completed phases

    def arrive(self):
        self.pending += 1
        if self.pending == self.count:
            self.pending = 0
            self.phases += 1

    def done(self, parity):
        # mbarrier try_wait.parity: true when the current phase's parity differs
        return (self.phases & 1) != parity


class Model:
    def __init__(self, rng, items, ring, double_s):
        self.rng = rng
        self.items = items  # steps per item, one persistent CTA
        self.R = ring
        self.ds = double_s
        B = Barrier
        self.str_full = [B(1) for _ in range(ring)]
        self.str_empty = [B(1) for _ in range(ring)]
        W = self.W = 2  # compute warps, each owning half of every buffer
        self.s_full = [B(1), B(1)]
        self.p_ready = [B(W), B(W)]
        self.dp_full, self.ds_ready = B(1), B(W)
        self.acc_done, self.acc_free, self.res_empty, self.res_full = B(1), B(W), B(1), B(1)
        self.queue = []  # tensor core: in-order products and commits
        self.loads = []  # tile loads in flight (complete in any order)
        self.slot_tile = [None] * ring  # step whose tiles a ring slot holds
        # [buffer][warp half]: ("S" or "P", step); [warp half]: ("dP" or "dS", step)
        self.sbuf = [[None] * W, [None] * W]
        self.dpbuf = [None] * W
        self.sbuf_consumed = [[True] * W, [True] * W]
        self.dp_consumed = [True] * W
        self.errors = []

    # --- helpers mirroring the kernel's
    def buf(self, g):
        return (g & 1) if self.ds else 0

    def spar(self, g):
        return ((g >> 1) & 1) if self.ds else (g & 1)

    def slot(self, pos):
        return pos % self.R

    def phase(self, pos):
        return (pos // self.R) & 1

    # --- the tensor core executes the head of its queue
    def tensor_step(self):
        kind, arg = self.queue.pop(0)
        if kind == "commit":
            arg.arrive()
            return
        op, g = kind, arg
        b = self.buf(g)
        for w in range(self.W):
            if op == "S":
                if self.sbuf[b][w] is not None and self.sbuf[b][w][0] == "P" \
                        and not self.sbuf_consumed[b][w]:
                    self.errors.append(f"S_{g} overwrote P_{self.sbuf[b][w][1]} before dV read it")
                self.sbuf[b][w] = ("S", g)
                self.sbuf_consumed[b][w] = False
            elif op == "dP":
                if self.dpbuf[w] is not None and self.dpbuf[w][0] == "dS" \
                        and not self.dp_consumed[w]:
                    self.errors.append(f"dP_{g} overwrote dS_{self.dpbuf[w][1]} before dK read it")
                self.dpbuf[w] = ("dP", g)
                self.dp_consumed[w] = False
            elif op == "dV":
                if self.sbuf[b][w] != ("P", g):
                    self.errors.append(f"dV_{g} read {self.sbuf[b][w]}")
                self.sbuf_consumed[b][w] = True
            elif op == "dK":
                if self.dpbuf[w] != ("dS", g):
                    self.errors.append(f"dK_{g} read {self.dpbuf[w]}")
                self.dp_consumed[w] = True
        if op in ("S", "dK") and self.slot_tile[self.slot(g)] != g:
            self.errors.append(f"{op}_{g} read the tiles of step {self.slot_tile[self.slot(g)]}")

    # --- roles as generators: each `yield cond` blocks until cond() holds
    def producer(self):
        sb = 0
        for t, n_steps in enumerate(self.items):
            for n in range(n_steps):
                pos = sb + n
                s = self.slot(pos)
                bar = self.str_empty[s]
                yield lambda b=bar, p=self.phase(pos) ^ 1: b.done(p)
                self.loads.append((s, pos))
                if n == 0 and t > 0:
                    yield lambda p=(t - 1) & 1: self.res_empty.done(p)
                if n == 0:
                    self.res_full.arrive()
            sb += n_steps

    def mma(self):
        sb = 0
        for t, n_steps in enumerate(self.items):
            yield lambda p=t & 1: self.res_full.done(p)
            yield lambda s=self.slot(sb), p=self.phase(sb): self.str_full[s].done(p)
            self.queue += [("S", sb), ("commit", self.s_full[self.buf(sb)]), ("dP", sb),
                           ("commit", self.dp_full)]
            for n in range(n_steps):
                g = sb + n
                more = n + 1 < n_steps
                if self.ds and more:  # the next step's scores first
                    yield lambda s=self.slot(g + 1), p=self.phase(g + 1): self.str_full[s].done(p)
                    self.queue += [("S", g + 1), ("commit", self.s_full[self.buf(g + 1)])]
                yield lambda b=self.buf(g), p=self.spar(g): self.p_ready[b].done(p)
                if n == 0 and t > 0:
                    yield lambda p=(t - 1) & 1: self.acc_free.done(p)
                self.queue.append(("dV", g))
                if not self.ds and more:
                    yield lambda s=self.slot(g + 1), p=self.phase(g + 1): self.str_full[s].done(p)
                    self.queue += [("S", g + 1), ("commit", self.s_full[0])]
                yield lambda p=g & 1: self.ds_ready.done(p)
                self.queue += [("dK", g), ("commit", self.str_empty[self.slot(g)])]
                if more:
                    self.queue += [("dP", g + 1), ("commit", self.dp_full)]
            self.queue += [("commit", self.acc_done), ("commit", self.res_empty)]
            sb += n_steps

    def compute(self, w):
        nb = 0
        for t, n_steps in enumerate(self.items):
            for n in range(n_steps):
                g = nb + n
                b = self.buf(g)
                yield lambda b=b, p=self.spar(g): self.s_full[b].done(p)
                if self.sbuf[b][w] != ("S", g):
                    self.errors.append(f"warp {w} step {g} read scores {self.sbuf[b][w]}")
                yield None  # the exponentials take a while
                self.sbuf[b][w] = ("P", g)
                self.sbuf_consumed[b][w] = False
                self.p_ready[b].arrive()
                yield lambda p=g & 1: self.dp_full.done(p)
                if self.dpbuf[w] != ("dP", g):
                    self.errors.append(f"warp {w} step {g} read dP {self.dpbuf[w]}")
                yield None
                self.dpbuf[w] = ("dS", g)
                self.dp_consumed[w] = False
                self.ds_ready.arrive()
            yield lambda p=t & 1: self.acc_done.done(p)
            yield None  # the epilogue
            self.acc_free.arrive()
            nb += n_steps

    def run(self):
        roles = {"producer": self.producer(), "mma": self.mma()}
        for w in range(self.W):
            roles[f"compute{w}"] = self.compute(w)
        waiting = {name: None for name in roles}
        finished = set()
        for _ in range(200000):
            enabled = []
            for name, gen in roles.items():
                if name in finished:
                    continue
                cond = waiting[name]
                if cond is None or cond():
                    enabled.append(name)
            if self.queue:
                enabled.append("tensor")
            if self.loads:
                enabled.append("tma")
            if not enabled:
                break
            pick = self.rng.choice(enabled)
            if pick == "tensor":
                self.tensor_step()
            elif pick == "tma":
                s, pos = self.loads.pop(self.rng.randrange(len(self.loads)))
                self.slot_tile[s] = pos
                self.str_full[s].arrive()
            else:
                try:
                    waiting[pick] = next(roles[pick])
                except StopIteration:
                    finished.add(pick)
                    waiting[pick] = None
        return finished == set(roles) and not self.queue and not self.loads


@pytest.mark.parametrize("double_s,ring", [(False, 2), (True, 4)], ids=["d128", "d64"])
def test_protocol_never_hangs_and_reads_its_own_step(double_s, ring):
    rng = random.Random(20261203 + ring)
    for trial in range(300):
        items = [rng.randint(1, 6) for _ in range(rng.randint(1, 4))]
        m = Model(rng, items, ring, double_s)
        assert m.run(), f"schedule {trial} (items {items}) hung"
        assert not m.errors, f"schedule {trial} (items {items}): {m.errors[:3]}"


def test_one_score_barrier_would_alias_at_d64():
    """The reason each score buffer has its own barriers: with one shared
    "scores ready" / "P ready" barrier and the next scores issued first, some
    schedule lets a barrier run two phases ahead, and a wait hangs."""

    class SharedBarriers(Model):
        def buf(self, g):  # the buffer still alternates ...
            return g & 1

        def spar(self, g):  # ... but every step waits on barrier [0]
            return g & 1

        def mma(self):
            self.s_full[1] = self.s_full[0]
            self.p_ready[1] = self.p_ready[0]
            yield from super().mma()

    rng = random.Random(7)
    hung = 0
    for _ in range(300):
        items = [rng.randint(2, 6) for _ in range(rng.randint(1, 3))]
        if not SharedBarriers(rng, items, 4, True).run():
            hung += 1
    assert hung > 0


@pytest.mark.parametrize("double_s,ring", [(False, 2), (True, 4)], ids=["d128", "d64"])
def test_model_sees_a_load_that_skips_the_empty_wait(double_s, ring):
    """The model itself is sensitive: a producer that reloads a ring slot
    without waiting for the products that read it is caught."""

    class EarlyLoad(Model):
        def producer(self):
            sb = 0
            for t, n_steps in enumerate(self.items):
                for n in range(n_steps):
                    pos = sb + n
                    self.loads.append((self.slot(pos), pos))
                    if n == 0 and t > 0:
                        yield lambda p=(t - 1) & 1: self.res_empty.done(p)
                    if n == 0:
                        self.res_full.arrive()
                    yield None
                sb += n_steps

    rng = random.Random(3)
    bad = 0
    for _ in range(100):
        items = [rng.randint(2, 6) for _ in range(rng.randint(1, 4))]
        m = EarlyLoad(rng, items, ring, double_s)
        bad += (not m.run()) or bool(m.errors)
    assert bad > 0


def test_model_sees_one_score_buffer_with_early_scores():
    """Issuing the next step's scores first into the same buffer overwrites a
    P that dV has not read; the model reports it."""

    class OneBuffer(Model):
        def buf(self, g):
            return 0

    rng = random.Random(5)
    bad = 0
    for _ in range(100):
        items = [rng.randint(2, 6) for _ in range(rng.randint(1, 4))]
        m = OneBuffer(rng, items, 4, True)
        bad += (not m.run()) or bool(m.errors)
    assert bad > 0


class FwdModel:
    """The forward kernel: one item is a pair of query tiles (groups 0 and 1,
    n0 and n1 key tiles, n0 <= n1), Q resident, K and V streamed through a
    two-stage ring, each group's scores and P in one tensor-memory buffer and
    its O accumulator in another; claimed items reach the other roles through
    a four-entry ring."""

    RING_ITEMS = 4

    def __init__(self, rng, items, warps=2):
        self.rng = rng
        self.items = items  # (n0, n1) per item of one persistent CTA
        self.W = W = warps  # warps per softmax group, each owning part of the rows
        B = Barrier
        self.q_full, self.q_empty = B(1), B(1)
        self.k_full, self.k_empty = [B(1), B(1)], [B(1), B(1)]
        self.v_full, self.v_empty = [B(1), B(1)], [B(1), B(1)]
        self.s_full = [B(1), B(1)]
        self.p_ready = [B(W), B(W)]
        self.pv_done = [B(1), B(1)]
        self.o_free = [B(W), B(W)]
        self.item_full = [B(1) for _ in range(self.RING_ITEMS)]
        self.item_ring = [None] * self.RING_ITEMS
        self.item_readers = [set() for _ in range(self.RING_ITEMS)]
        self.n_readers = 1 + 2 * W  # the issuer and every softmax warp
        self.queue, self.loads = [], []
        self.q_tile = None
        self.k_tile, self.v_tile = [None, None], [None, None]
        # per group and warp: ("S" | "P", item, tile) and (item, PV products in O)
        self.sbuf = [[None] * W for _ in range(2)]
        self.p_read = [[True] * W for _ in range(2)]
        self.obuf = [[None] * W for _ in range(2)]
        self.o_read = [[True] * W for _ in range(2)]
        self.errors = []

    @staticmethod
    def slot(pos):
        return pos % 2

    @staticmethod
    def phase(pos):
        return (pos // 2) & 1

    def tensor_step(self):
        kind, *arg = self.queue.pop(0)
        if kind == "commit":
            arg[0].arrive()
            return
        g, pos, t, j = arg[:4]
        if kind == "S":
            if self.q_tile != t:
                self.errors.append(f"S{g} of item {t} read the Q of item {self.q_tile}")
            if self.k_tile[self.slot(pos)] != pos:
                self.errors.append(f"S{g} at {pos} read the K tile {self.k_tile[self.slot(pos)]}")
            for w in range(self.W):
                if not self.p_read[g][w]:
                    self.errors.append(f"S{g}({t},{j}) overwrote a P before P V read it")
                self.sbuf[g][w] = ("S", t, j)
        else:  # "PV"
            first = arg[4]
            if self.v_tile[self.slot(pos)] != pos:
                self.errors.append(f"PV{g} at {pos} read the V tile {self.v_tile[self.slot(pos)]}")
            for w in range(self.W):
                if self.sbuf[g][w] != ("P", t, j):
                    self.errors.append(f"PV{g}({t},{j}) read {self.sbuf[g][w]}")
                self.p_read[g][w] = True
                if first:
                    if not self.o_read[g][w]:
                        self.errors.append(f"PV{g} of item {t} overwrote an O not yet stored")
                    self.obuf[g][w] = (t, 1)
                    self.o_read[g][w] = False
                elif self.obuf[g][w] != (t, j):
                    self.errors.append(f"PV{g}({t},{j}) accumulated into {self.obuf[g][w]}")
                else:
                    self.obuf[g][w] = (t, j + 1)

    def publish(self, t, item):
        r = t % self.RING_ITEMS
        if t >= self.RING_ITEMS and len(self.item_readers[r]) < self.n_readers:
            self.errors.append(f"item ring entry {r} overwritten before every role read it")
        self.item_ring[r] = item
        self.item_readers[r] = set()
        self.item_full[r].arrive()

    def claim(self, t, who):
        r = t % self.RING_ITEMS
        yield lambda: self.item_full[r].done((t // self.RING_ITEMS) & 1)
        self.item_readers[r].add(who)
        return self.item_ring[r]

    def producer(self):
        kvb = 0
        for t, item in enumerate(self.items + [None]):
            self.publish(t, item)
            if item is None:
                return
            n0, n1 = item
            if t == 0 and n1 > 0:
                self.loads.append(("Q", t))
            for j in range(n1):
                pos = kvb + j
                s, ph = self.slot(pos), self.phase(pos)
                yield lambda s=s, p=ph ^ 1: self.k_empty[s].done(p)
                self.loads.append(("K", pos))
                if j == 0 and t > 0:
                    yield lambda p=(t - 1) & 1: self.q_empty.done(p)
                    self.loads.append(("Q", t))
                yield lambda s=s, p=ph ^ 1: self.v_empty[s].done(p)
                self.loads.append(("V", pos))
            kvb += n1

    def land(self, load):
        kind, x = load
        if kind == "Q":
            self.q_tile = x
            self.q_full.arrive()
        elif kind == "K":
            self.k_tile[self.slot(x)] = x
            self.k_full[self.slot(x)].arrive()
        else:
            self.v_tile[self.slot(x)] = x
            self.v_full[self.slot(x)].arrive()

    def mma(self):
        kvb = base0 = base1 = 0
        for t in range(len(self.items) + 1):
            item = yield from self.claim(t, "mma")
            if item is None:
                return
            n0, n1 = item
            if n1 == 0:  # a block-sparse item without key tiles (a CTA's only item)
                continue
            yield lambda p=t & 1: self.q_full.done(p)
            yield lambda s=self.slot(kvb), p=self.phase(kvb): self.k_full[s].done(p)
            self.queue += [("S", 0, kvb, t, 0), ("commit", self.s_full[0]),
                           ("S", 1, kvb, t, 0), ("commit", self.s_full[1]),
                           ("commit", self.k_empty[self.slot(kvb)])]
            for j in range(n1):
                pos = kvb + j
                s, ph = self.slot(pos), self.phase(pos)
                sn, phn = self.slot(pos + 1), self.phase(pos + 1)
                pre1 = False
                if j < n0:
                    yield lambda p=(base0 + j) & 1: self.p_ready[0].done(p)
                    yield lambda: self.v_full[s].done(ph)
                    if j == 0 and t > 0:
                        yield lambda p=(t - 1) & 1: self.o_free[0].done(p)
                    if j + 1 < n1:
                        yield lambda: self.k_full[sn].done(phn)
                    self.queue += [("PV", 0, pos, t, j, j == 0), ("commit", self.pv_done[0])]
                    if j + 1 < n0:
                        self.queue.append(("S", 0, pos + 1, t, j + 1))
                    yield None  # the issue takes a while; the others move meanwhile
                    pre1 = self.p_ready[1].done((base1 + j) & 1) and (
                        j > 0 or t == 0 or self.o_free[1].done((t - 1) & 1))
                    if j + 1 < n0:
                        self.queue.append(("commit", self.s_full[0]))
                if not pre1:
                    yield lambda p=(base1 + j) & 1: self.p_ready[1].done(p)
                    if j >= n0:
                        yield lambda: self.v_full[s].done(ph)
                    if j == 0 and t > 0:
                        yield lambda p=(t - 1) & 1: self.o_free[1].done(p)
                    if j >= n0 and j + 1 < n1:
                        yield lambda: self.k_full[sn].done(phn)
                self.queue += [("PV", 1, pos, t, j, j == 0), ("commit", self.v_empty[s])]
                if j + 1 < n1:
                    self.queue.append(("S", 1, pos + 1, t, j + 1))
                self.queue.append(("commit", self.pv_done[1]))
                if j + 1 < n1:
                    self.queue += [("commit", self.s_full[1]), ("commit", self.k_empty[sn])]
            self.queue.append(("commit", self.q_empty))
            kvb += n1
            base0 += n0
            base1 += n1

    def softmax(self, g, w):
        tb = 0
        for t in range(len(self.items) + 1):
            item = yield from self.claim(t, ("softmax", g, w))
            if item is None:
                return
            nkv = item[g]
            for j in range(nkv):
                yield lambda p=(tb + j) & 1: self.s_full[g].done(p)
                if self.sbuf[g][w] != ("S", t, j):
                    self.errors.append(f"softmax {g}.{w} at ({t},{j}) read {self.sbuf[g][w]}")
                yield None  # the exponentials
                if j > 0 and self.obuf[g][w] != (t, j):  # the lazy rescale of O
                    self.errors.append(f"softmax {g}.{w} rescaled O {self.obuf[g][w]} at ({t},{j})")
                yield None
                if j > 0 and self.obuf[g][w] != (t, j):
                    self.errors.append(f"O {g}.{w} changed under the rescale at ({t},{j})")
                self.sbuf[g][w] = ("P", t, j)
                self.p_read[g][w] = False
                self.p_ready[g].arrive()
            if nkv > 0:
                yield lambda p=(tb + nkv - 1) & 1: self.pv_done[g].done(p)
                if self.obuf[g][w] != (t, nkv):
                    self.errors.append(f"epilogue {g}.{w} of item {t} read O {self.obuf[g][w]}")
                yield None  # the stores
                if self.obuf[g][w] != (t, nkv):
                    self.errors.append(f"O {g}.{w} changed under the epilogue of item {t}")
                self.o_read[g][w] = True
            self.o_free[g].arrive()
            tb += nkv

    def run(self):
        roles = {"producer": self.producer(), "mma": self.mma()}
        for g in range(2):
            for w in range(self.W):
                roles[("softmax", g, w)] = self.softmax(g, w)
        waiting = {name: None for name in roles}
        finished = set()
        for _ in range(400000):
            enabled = [n for n in roles if n not in finished
                       and (waiting[n] is None or waiting[n]())]
            if self.queue:
                enabled.append("tensor")
            if self.loads:
                enabled.append("tma")
            if not enabled:
                break
            pick = self.rng.choice(enabled)
            if pick == "tensor":
                self.tensor_step()
            elif pick == "tma":
                self.land(self.loads.pop(self.rng.randrange(len(self.loads))))
            else:
                try:
                    waiting[pick] = next(roles[pick])
                except StopIteration:
                    finished.add(pick)
                    waiting[pick] = None
        return finished == set(roles) and not self.queue and not self.loads


def fwd_items(rng, causal):
    out = []
    for _ in range(rng.randint(1, 5)):
        n0 = rng.randint(1, 6)
        out.append((n0, n0 + (rng.random() < 0.7)) if causal else (n0, n0))
    return out


@pytest.mark.parametrize("causal", [True, False], ids=["causal", "full"])
def test_forward_protocol_never_hangs_and_reads_its_own_tile(causal):
    rng = random.Random(20261204 + causal)
    for trial in range(300):
        items = fwd_items(rng, causal)
        m = FwdModel(rng, items)
        assert m.run(), f"schedule {trial} (items {items}) hung"
        assert not m.errors, f"schedule {trial} (items {items}): {m.errors[:3]}"


def test_forward_single_block_sparse_items():
    """A block-sparse CTA runs one item with n0 = n1 key tiles, none at all
    included (both groups store O = 0 and free their accumulators)."""
    rng = random.Random(11)
    for n in [0, 1, 2, 5]:
        for _ in range(50):
            m = FwdModel(rng, [(n, n)])
            assert m.run() and not m.errors, (n, m.errors[:3])


def test_forward_model_sees_scores_committed_before_p_is_read():
    """Sensitivity: a group's next scores issued before its P V (the order
    the bursts exist to keep) overwrite a P that P V has not read."""

    class EarlyScores(FwdModel):
        def mma(self):
            for cond in super().mma():
                # move every "S" of group 0 ahead of the "PV" queued just before it
                q = self.queue
                for i in range(1, len(q)):
                    if q[i][0] == "S" and q[i][1] == 0 and q[i - 1][0] == "commit" \
                            and i >= 2 and q[i - 2][0] == "PV" and q[i - 2][1] == 0:
                        q[i - 2], q[i] = q[i], q[i - 2]
                yield cond

    rng = random.Random(13)
    bad = 0
    for _ in range(100):
        m = EarlyScores(rng, fwd_items(rng, True))
        bad += (not m.run()) or bool(m.errors)
    assert bad > 0


class DecodeModel:
    """The decode kernel's split: one item (n key tiles of one head and key
    range), one softmax warp, Q resident, K and V streamed through a ring of
    `stages`, two score buffers (tile t in buffer t & 1, each with its own
    scores-ready barrier) and the next-but-one tile's scores issued after the
    P V that frees their buffer."""

    def __init__(self, rng, n, stages):
        self.rng, self.n, self.R = rng, n, stages
        B = Barrier
        self.q_full = B(1)
        self.k_full, self.k_empty = [B(1) for _ in range(stages)], [B(1) for _ in range(stages)]
        self.v_full, self.v_empty = [B(1) for _ in range(stages)], [B(1) for _ in range(stages)]
        self.s_full = [B(1), B(1)]
        self.p_ready, self.pv_done = B(1), B(1)
        self.queue, self.loads = [], []
        self.q_in = False
        self.k_tile, self.v_tile = [None] * stages, [None] * stages
        self.sbuf = [None, None]  # ("S" | "P", tile)
        self.p_read = [True, True]
        self.o = 0  # P V products accumulated
        self.errors = []

    def tensor_step(self):
        kind, *arg = self.queue.pop(0)
        if kind == "commit":
            arg[0].arrive()
            return
        t = arg[0]
        b, st = t & 1, t % self.R
        if kind == "S":
            if not self.q_in or self.k_tile[st] != t:
                self.errors.append(f"S({t}) read K tile {self.k_tile[st]}")
            if not self.p_read[b]:
                self.errors.append(f"S({t}) overwrote P{self.sbuf[b]} before P V read it")
            self.sbuf[b] = ("S", t)
        else:  # PV
            if self.sbuf[b] != ("P", t) or self.v_tile[st] != t:
                self.errors.append(f"PV({t}) read {self.sbuf[b]}, V tile {self.v_tile[st]}")
            if self.o != t:
                self.errors.append(f"PV({t}) accumulated onto {self.o} products")
            self.p_read[b] = True
            self.o = t + 1

    def producer(self):
        self.loads.append(("Q", 0))
        for t in range(self.n):
            st, ph = t % self.R, (t // self.R) & 1
            yield lambda st=st, ph=ph: self.k_empty[st].done(ph ^ 1)
            self.loads.append(("K", t))
            yield lambda st=st, ph=ph: self.v_empty[st].done(ph ^ 1)
            self.loads.append(("V", t))

    def land(self, load):
        kind, t = load
        if kind == "Q":
            self.q_in = True
            self.q_full.arrive()
        elif kind == "K":
            self.k_tile[t % self.R] = t
            self.k_full[t % self.R].arrive()
        else:
            self.v_tile[t % self.R] = t
            self.v_full[t % self.R].arrive()

    def issue_s(self, t):
        self.queue += [("S", t), ("commit", self.s_full[t & 1]),
                       ("commit", self.k_empty[t % self.R])]

    def mma(self):
        yield lambda: self.q_full.done(0)
        yield lambda: self.k_full[0].done(0)
        self.issue_s(0)
        if self.n > 1:
            yield lambda: self.k_full[1 % self.R].done((1 // self.R) & 1)
            self.issue_s(1)
        for t in range(self.n):
            yield lambda t=t: self.p_ready.done(t & 1)
            yield lambda t=t: self.v_full[t % self.R].done((t // self.R) & 1)
            self.queue += [("PV", t), ("commit", self.pv_done),
                           ("commit", self.v_empty[t % self.R])]
            if t + 2 < self.n:
                u = t + 2
                yield lambda u=u: self.k_full[u % self.R].done((u // self.R) & 1)
                self.issue_s(u)

    def softmax(self):
        for t in range(self.n):
            yield lambda t=t: self.s_full[t & 1].done((t >> 1) & 1)
            if self.sbuf[t & 1] != ("S", t):
                self.errors.append(f"softmax {t} read {self.sbuf[t & 1]}")
            yield None
            self.sbuf[t & 1] = ("P", t)
            self.p_read[t & 1] = False
            if t > 0:  # P V of the previous tile done before O is rescaled
                yield lambda t=t: self.pv_done.done((t - 1) & 1)
                if self.o != t:
                    self.errors.append(f"softmax {t} rescaled O with {self.o} products")
                yield None
                if self.o != t:
                    self.errors.append(f"O changed under the rescale at {t}")
            self.p_ready.arrive()
        yield lambda: self.pv_done.done((self.n - 1) & 1)
        if self.o != self.n:
            self.errors.append(f"epilogue read O with {self.o} of {self.n} products")

    def run(self):
        roles = {"producer": self.producer(), "mma": self.mma(), "softmax": self.softmax()}
        waiting = {name: None for name in roles}
        finished = set()
        for _ in range(100000):
            enabled = [r for r in roles if r not in finished
                       and (waiting[r] is None or waiting[r]())]
            if self.queue:
                enabled.append("tensor")
            if self.loads:
                enabled.append("tma")
            if not enabled:
                break
            pick = self.rng.choice(enabled)
            if pick == "tensor":
                self.tensor_step()
            elif pick == "tma":
                self.land(self.loads.pop(self.rng.randrange(len(self.loads))))
            else:
                try:
                    waiting[pick] = next(roles[pick])
                except StopIteration:
                    finished.add(pick)
                    waiting[pick] = None
        return finished == set(roles) and not self.queue and not self.loads


@pytest.mark.parametrize("stages", [2, 4], ids=["d128", "d64"])
def test_decode_protocol_never_hangs_and_reads_its_own_tile(stages):
    rng = random.Random(20261205 + stages)
    for trial in range(300):
        n = rng.randint(1, 9)
        m = DecodeModel(rng, n, stages)
        assert m.run(), f"schedule {trial} (n = {n}) hung"
        assert not m.errors, f"schedule {trial} (n = {n}): {m.errors[:3]}"


def test_decode_model_sees_scores_issued_into_a_busy_buffer():
    """Sensitivity: issuing tile t + 2's scores before P V(t) overwrites P(t)."""

    class Early(DecodeModel):
        def mma(self):
            yield lambda: self.q_full.done(0)
            yield lambda: self.k_full[0].done(0)
            self.issue_s(0)
            if self.n > 1:
                yield lambda: self.k_full[1 % self.R].done((1 // self.R) & 1)
                self.issue_s(1)
            for t in range(self.n):
                if t + 2 < self.n:
                    u = t + 2
                    yield lambda u=u: self.k_full[u % self.R].done((u // self.R) & 1)
                    self.issue_s(u)
                yield lambda t=t: self.p_ready.done(t & 1)
                yield lambda t=t: self.v_full[t % self.R].done((t // self.R) & 1)
                self.queue += [("PV", t), ("commit", self.pv_done),
                               ("commit", self.v_empty[t % self.R])]

    rng = random.Random(17)
    bad = 0
    for _ in range(100):
        m = Early(rng, rng.randint(3, 9), 4)
        bad += (not m.run()) or bool(m.errors)
    assert bad > 0
