"""Models of the mbarrier protocols of two tensor-core kernels, run under random timing.

Each model lists, per role of one CTA, the barrier operations the kernel performs in program
order: waits (for phase k of a barrier, by parity k & 1, exactly as the kernels call
mbarrier.try_wait.parity), arrivals, and products whose commits arrive later.  A scheduler
interleaves the roles at random and completes TMA copies in any order and products in
issue order.  A wait passes iff the barrier's completed-phase count has the other parity,
which is what the hardware checks; the model reports

  * premature: a wait passed before the phase it stands for had completed (the barrier
    was two phases behind), and
  * deadlock: no role can move (in particular a wait whose phase completed but whose
    parity came round again, the barrier being two phases ahead), and
  * hazard: a ('check', predicate, what) step found the model state wrong, e.g. the query
    tile rewritten in TMEM while a product that reads the old one was still pending.

Models: the paired head-dimension-128 forward (fa_tc.cu: two query tiles, P written over S,
O final once the next S is complete), the head-dimension-32/64 forward (P in TMEM columns of
its own, S released to the next product once read), the head-dimension-256 forward (fa_tc256.cu: S double-buffered, O += P V, the
conditional O rescale, the next item's query tile written on the last step, the per-item
epilogue) and the head-dimension-256 backward
(fa_bwd256.cu: the dQ / dK template and the dV kernel with its two S^T buffers and
rings), and the head-dimension-32-128 backward (fa_bwd.cu: the dQ kernel and the dK/dV
kernel, whose elementwise warps stage their per-column vectors without a barrier across
warps).  A change to either kernel's barrier order must be mirrored here.  Planted
mistakes (the epilogue's two waits in a row; the next query tile written before the last
S product is seen complete; a single-buffered dV hand-over) must fail.
"""
import random

import pytest


class Model:
    """Barriers with arrival counts; roles as lists of operations; random interleaving."""

    def __init__(self, seed):
        self.rnd = random.Random(seed)
        self.need, self.got, self.done = {}, {}, {}

    def bar(self, name, count=1):
        self.need[name], self.got[name], self.done[name] = count, 0, 0

    def arrive(self, name):
        self.got[name] += 1
        if self.got[name] == self.need[name]:
            self.got[name] = 0
            self.done[name] += 1

    def run(self, roles, max_moves=200000):
        """roles: name -> list of ('wait', bar, phase) | ('arrive', bar) |
        ('copy', bar) (completes later, any order) | ('mma', [bars]) (commits later, in
        order) | ('group', tag) (named barrier of the roles sharing tag).  Returns 'ok',
        'premature ...', 'deadlock ...' or 'hazard ...'."""
        pc = {r: 0 for r in roles}
        copies, pipe = [], []
        group_count = {}
        for _ in range(max_moves):
            ready = []
            for r, prog in roles.items():
                if pc[r] >= len(prog):
                    continue
                op = prog[pc[r]]
                if op[0] == "wait":
                    name, k = op[1], op[2]
                    if (self.done[name] & 1) != (k & 1):
                        if self.done[name] < k + 1:
                            return "premature %s phase %d (completed %d)" % (name, k, self.done[name])
                        ready.append(r)
                elif op[0] == "group":
                    tag, n = op[1], op[2]
                    members = [x for x in roles if x.startswith(tag)]
                    # passes when every member has reached this instance (or gone past it)
                    if all(group_count.get(x, 0) > n or
                           (pc[x] < len(roles[x]) and roles[x][pc[x]][:2] == ("group", tag)
                            and roles[x][pc[x]][2] == n) for x in members):
                        ready.append(r)
                else:
                    ready.append(r)
            if copies:
                ready.append("copy")
            if pipe:
                ready.append("pipe")
            if not ready:
                if all(pc[r] >= len(p) for r, p in roles.items()) and not copies and not pipe:
                    return "ok"
                return "deadlock " + str({r: roles[r][pc[r]] if pc[r] < len(roles[r]) else "end"
                                          for r in roles})
            r = self.rnd.choice(ready)
            if r == "copy":
                self.arrive(copies.pop(self.rnd.randrange(len(copies))))
                continue
            if r == "pipe":
                for name in pipe.pop(0):
                    self.arrive(name)
                continue
            op = roles[r][pc[r]]
            if op[0] == "check":
                if not op[1](self):
                    return "hazard " + op[2]
            elif op[0] == "arrive":
                self.arrive(op[1])
            elif op[0] == "copy":
                copies.append(op[1])
            elif op[0] == "mma":
                pipe.append(list(op[1]))
            elif op[0] == "group":
                group_count[r] = group_count.get(r, 0) + 1
            pc[r] += 1
        return "no end"


# ----------------------------------------------------------------- D = 128 forward, paired tiles
def tc128_roles(m, items, s_before_pv=False):
    """fa_tc.cu's paired schedule where P overwrites S, one CTA over `items` ((nA, nB) key
    tiles per item); loads are taken as ready.  The softmax of a tile waits only for S: the
    commit behind s_full tracks every product the MMA thread issued before S(j), so
    O += P(j-1) V(j-1) is complete too, which a check step asserts before O is touched.
    Its epilogue waits once, for the tile's last O product.  s_before_pv plants an issue
    order with S(j+1) ahead of O += P(j) V(j)."""
    for t in "AB":
        m.bar(("s_full", t))
        m.bar(("p_full", t))
        m.bar(("o_done", t))
    mma = []
    for nA, nB in items:
        n = {"A": nA, "B": nB}
        for t in "AB":
            mma.append(("mma", [("s_full", t)]))
        for j in range(max(nA, nB)):
            for t in "AB":
                pv = [("wait", ("p_full", t), None), ("mma", [("o_done", t)])] if j < n[t] else []
                s_next = [("mma", [("s_full", t)])] if j + 1 < n[t] else []
                mma.extend(s_next + pv if s_before_pv else pv + s_next)
    # the MMA's p_full waits count per tile
    cnt = {"A": 0, "B": 0}
    for k, op in enumerate(mma):
        if op[0] == "wait":
            t = op[1][1]
            mma[k] = ("wait", op[1], cnt[t])
            cnt[t] += 1
    roles = {"mma": mma}
    for t in "AB":
        sm, s_cnt, o_base = [], 0, 0
        for nA, nB in items:
            n = nA if t == "A" else nB
            for j in range(n):
                sm.append(("wait", ("s_full", t), s_cnt))
                s_cnt += 1
                if j > 0:
                    need = o_base + j   # O += P(j-1) V(j-1) of this item complete
                    sm.append(("check", lambda mm, t=t, need=need: mm.done[("o_done", t)] >= need,
                               "tile %s read O before its last product completed" % t))
                sm.append(("arrive", ("p_full", t)))
            sm.append(("wait", ("o_done", t), o_base + n - 1))
            o_base += n
        roles["softmax_" + t] = sm
    return roles


def test_tc128_paired_protocol():
    for seed in range(400):
        m = Model(seed)
        items = [(m.rnd.randint(1, 5), m.rnd.randint(1, 5)) for _ in range(m.rnd.randint(1, 4))]
        res = m.run(tc128_roles(m, items))
        assert res == "ok", (seed, items, res)


def test_tc128_planted_s_before_pv_fails():
    bad = 0
    for seed in range(200):
        m = Model(seed)
        items = [(m.rnd.randint(2, 5), m.rnd.randint(2, 5)) for _ in range(m.rnd.randint(1, 3))]
        bad += m.run(tc128_roles(m, items, s_before_pv=True)) != "ok"
    assert bad > 0


# ----------------------------------------------------------------- D <= 64 forward, P apart
def tc_sep_roles(m, items, no_s_read_wait=False):
    """fa_tc.cu's paired schedule where P has TMEM columns of its own (D <= 64): each tile's
    next S product waits only until the softmax has read the current S (s_read), ahead of
    O += P V; the softmax waits for the previous O product before it stores P (which that
    product reads) and before O is rescaled.  Checks: S(j) is still in its region when it is
    read, and the previous O product is complete when P is stored.  no_s_read_wait plants an
    MMA issuer that overwrites S without waiting for the read."""
    for t in "AB":
        for b in ("s_full", "s_read", "p_full", "o_done"):
            m.bar((b, t))
    mma, issued, sr, pc = [], {"A": 0, "B": 0}, {"A": 0, "B": 0}, {"A": 0, "B": 0}

    def issue_s(t):
        if issued[t] > 0 and not no_s_read_wait:
            mma.append(("wait", ("s_read", t), sr[t]))
            sr[t] += 1
        mma.append(("mma", [("s_full", t)]))
        issued[t] += 1

    for nA, nB in items:
        n = {"A": nA, "B": nB}
        for t in "AB":
            issue_s(t)
        for j in range(max(nA, nB)):
            for t in "AB":
                if j + 1 < n[t]:
                    issue_s(t)
            for t in "AB":
                if j < n[t]:
                    mma.append(("wait", ("p_full", t), pc[t]))
                    pc[t] += 1
                    mma.append(("mma", [("o_done", t)]))
    roles = {"mma": mma}
    for t in "AB":
        sm, s_cnt, o_cnt = [], 0, 0
        for nA, nB in items:
            n = nA if t == "A" else nB
            o_base = o_cnt
            for j in range(n):
                sm.append(("wait", ("s_full", t), s_cnt))
                s_cnt += 1
                sm.append(("check", lambda mm, t=t, k=s_cnt: mm.done[("s_full", t)] == k,
                           "tile %s S overwritten before it was read" % t))
                sm.append(("arrive", ("s_read", t)))
                if j > 0:
                    sm.append(("wait", ("o_done", t), o_cnt))
                    o_cnt += 1
                    sm.append(("check", lambda mm, t=t, k=o_base + j: mm.done[("o_done", t)] >= k,
                               "tile %s P stored before the last O product read it" % t))
                sm.append(("arrive", ("p_full", t)))
            sm.append(("wait", ("o_done", t), o_cnt))
            o_cnt += 1
        roles["softmax_" + t] = sm
    return roles


def test_tc_sep_protocol():
    for seed in range(400):
        m = Model(seed)
        items = [(m.rnd.randint(1, 5), m.rnd.randint(1, 5)) for _ in range(m.rnd.randint(1, 4))]
        res = m.run(tc_sep_roles(m, items))
        assert res == "ok", (seed, items, res)


def test_tc_sep_planted_missing_s_read_fails():
    bad = 0
    for seed in range(200):
        m = Model(seed)
        items = [(m.rnd.randint(2, 5), m.rnd.randint(2, 5)) for _ in range(m.rnd.randint(1, 3))]
        bad += m.run(tc_sep_roles(m, items, no_s_read_wait=True)).startswith("hazard")
    assert bad > 0


# ----------------------------------------------------------------- D = 256 forward
def tc256_roles(m, items, rescale_prob, two_epilogue_waits=False, early_q=False):
    """fa_tc256.cu, one CTA over `items` (key steps per item); loads are taken as ready.
    The softmax writes a CTA's first query tile into TMEM at the start and every later one
    on the previous item's last step, after that step's S product (the last to read the old
    tile) is seen complete; a check step asserts exactly that.  early_q plants the write
    before that wait."""
    for b in (0, 1):
        m.bar(("s_full", b))
        m.bar(("p_full", b))
    m.bar("o_done")
    m.bar("q_ready")
    mma, sm = [], []
    g = 0
    for it, nkv in enumerate(items):
        mma.append(("wait", "q_ready", it))
        mma.append(("mma", [("s_full", g & 1)]))
        if nkv > 1:
            mma.append(("mma", [("s_full", (g + 1) & 1)]))
        for j in range(nkv):
            gj = g + j
            mma.append(("wait", ("p_full", gj & 1), gj >> 1))
            mma.append(("mma", ["o_done"]))
            if j + 2 < nkv:
                mma.append(("mma", [("s_full", (gj + 2) & 1)]))
        g += nkv
    g = pv = 0

    def s_done_through(n):   # every S product of the first n steps is complete
        return lambda mm: mm.done[("s_full", 0)] + mm.done[("s_full", 1)] >= n

    for it, nkv in enumerate(items):
        if it == 0:
            sm.append(("arrive", "q_ready"))
        for j in range(nkv):
            gj = g + j
            last_with_next = j + 1 == nkv and it + 1 < len(items)
            if early_q and last_with_next:
                sm.append(("check", s_done_through(g + nkv), "query tile rewritten early"))
                sm.append(("arrive", "q_ready"))
            sm.append(("wait", ("s_full", gj & 1), gj >> 1))
            resc = j > 0 and m.rnd.random() < rescale_prob
            last_sync = (j > 0 and j + 1 == nkv) and not two_epilogue_waits
            if resc or last_sync:
                sm.append(("wait", "o_done", pv + j - 1))
            sm.append(("arrive", ("p_full", gj & 1)))
            if last_with_next and not early_q:
                # the next item's query tile into TMEM, then q_ready
                sm.append(("check", s_done_through(g + nkv), "query tile rewritten early"))
                sm.append(("arrive", "q_ready"))
        pv += nkv
        if two_epilogue_waits and nkv >= 2:
            sm.append(("wait", "o_done", pv - 2))
        sm.append(("wait", "o_done", pv - 1))
        g += nkv
    return {"mma": mma, "softmax": sm}


@pytest.mark.parametrize("rescale_prob", [0.0, 0.5, 1.0])
def test_tc256_forward_protocol(rescale_prob):
    for seed in range(300):
        m = Model(seed)
        items = [m.rnd.randint(1, 6) for _ in range(m.rnd.randint(1, 4))]
        res = m.run(tc256_roles(m, items, rescale_prob))
        assert res == "ok", (seed, items, res)


def test_tc256_planted_early_query_write_fails():
    # writing the next query tile before the item's last S product is seen complete
    bad = 0
    for seed in range(300):
        m = Model(seed)
        items = [m.rnd.randint(1, 4) for _ in range(m.rnd.randint(2, 4))]
        res = m.run(tc256_roles(m, items, 0.5, early_q=True))
        bad += res.startswith("hazard")
    assert bad > 0


def test_tc256_planted_two_epilogue_waits_fail():
    # waiting for the last two products one after the other misreads the parity when both
    # completed before the first wait
    bad = 0
    for seed in range(300):
        m = Model(seed)
        items = [m.rnd.randint(2, 6) for _ in range(m.rnd.randint(1, 4))]
        bad += m.run(tc256_roles(m, items, 0.5, two_epilogue_waits=True)) != "ok"
    assert bad > 0


# ----------------------------------------------------------------- D = 256 backward
def bwd256_roles(m, role, n, slots, single_buffer_dv=False):
    """fa_bwd256.cu, one CTA: role 'dq' / 'dk' (one template) or 'dv'; n streamed
    sub-tiles; two elementwise warp groups (ew0, ew1) standing for the eight warps."""
    fixed = role != "dv"
    m.bar("fixed")
    for s in range(slots):
        m.bar(("full", s))
        m.bar(("empty", s))
    for b in (0, 1):
        m.bar(("s", b))
        m.bar(("x", b), 2)
    m.bar("dp")
    m.bar("ds", 2)
    m.bar("row")
    m.bar("done")
    slot = lambda pos: pos % slots
    fill = lambda pos: pos // slots
    # the loader's order of streamed sub-tiles (after the row tile's two halves)
    if role != "dv":
        order = [("X" if k % 2 == 0 else "Y", k // 2) for k in range(2 * n)]
    else:
        order = [("X", 0)] + ([("X", 1)] if n > 1 else [])
        for s in range(n):
            order.append(("Y", s))
            if s + 2 < n:
                order.append(("X", s + 2))
    pos_of = {o: 2 + i for i, o in enumerate(order)}
    load = [("copy", "fixed")] if fixed else []
    for pos in range(2 + 2 * n):
        if pos >= slots:
            load.append(("wait", ("empty", slot(pos)), fill(pos) - 1))
        load.append(("copy", ("full", slot(pos))))
    mma = [("wait", "fixed", 0)] if fixed else []
    mma.append(("wait", "row", 0))

    def full(o):
        p = pos_of[o]
        return ("wait", ("full", slot(p)), fill(p))

    if role != "dv":
        def issue_s(j):
            mma.extend([full(("X", j)), ("mma", [("s", 0)])])

        def issue_dp(j):
            mma.extend([full(("Y", j)), ("mma", ["dp", ("empty", slot(pos_of[("Y", j)]))])])

        issue_s(0)
        issue_dp(0)
        for j in range(n):
            mma.append(("wait", ("x", 0), j))
            if j + 1 < n:
                issue_s(j + 1)
            mma.append(("wait", "ds", j))
            mma.append(("mma", [("empty", slot(pos_of[("X", j)]))]))
            if j + 1 < n:
                issue_dp(j + 1)
    else:
        def issue_s(s):
            b = 0 if single_buffer_dv else s & 1
            mma.extend([full(("X", s)), ("mma", [("s", b), ("empty", slot(pos_of[("X", s)]))])])

        issue_s(0)
        if n > 1:
            issue_s(1)
        for s in range(n):
            if single_buffer_dv:
                mma.append(("wait", ("x", 0), s))
            else:
                mma.append(("wait", ("x", s & 1), s >> 1))
            mma.extend([full(("Y", s)), ("mma", [("empty", slot(pos_of[("Y", s)]))])])
            if s + 2 < n:
                issue_s(s + 2)
    mma.append(("mma", ["done"]))

    def ew(first):
        e = [("wait", "fixed", 0)] if role == "dq" else []
        e += [("wait", ("full", slot(0)), 0), ("wait", ("full", slot(1)), 0), ("group", "ew", 0)]
        if first:
            e += [("arrive", ("empty", slot(0))), ("arrive", ("empty", slot(1))), ("arrive", "row")]
        k = 1
        for j in range(n):
            if role == "dv":
                if single_buffer_dv:
                    e.append(("wait", ("s", 0), j))
                else:
                    e.append(("wait", ("s", j & 1), j >> 1))
                e.append(("group", "ew", k)); k += 1
                e.append(("arrive", ("x", 0 if single_buffer_dv else j & 1)))
            else:
                e.append(("wait", ("s", 0), j))
                if role == "dk":
                    e.append(("group", "ew", k)); k += 1
                e.append(("arrive", ("x", 0)))
                e.append(("wait", "dp", j))
                e.append(("arrive", "ds"))
        e.append(("wait", "done", 0))
        return e

    return {"load": load, "mma": mma, "ew0": ew(True), "ew1": ew(False)}


@pytest.mark.parametrize("role,slots", [("dq", 5), ("dk", 5), ("dv", 6)])
@pytest.mark.parametrize("n", [1, 2, 3, 5, 8])
def test_bwd256_protocol(role, slots, n):
    for seed in range(60):
        m = Model(seed)
        res = m.run(bwd256_roles(m, role, n, slots))
        assert res == "ok", (role, n, seed, res)


def test_bwd256_planted_single_buffered_dv_fails():
    bad = 0
    for seed in range(60):
        m = Model(seed)
        bad += m.run(bwd256_roles(m, "dv", 4, 6, single_buffer_dv=True)) != "ok"
    assert bad > 0


# ----------------------------------------------------------------- D <= 128 backward
def bwd_dq_roles(m, n, no_ds_free_wait=False):
    """fa_bwd.cu's dQ kernel, one CTA over n key tiles; loads taken as ready; two
    elementwise groups stand for the eight warps (each barrier they arrive on counts both).
    S(j+1) is issued once S(j) is read (x_ready), dP(j+1) once dP(j) is read (dp_free), and
    dQ += dS K_j once dS is stored (ds_ready); the elementwise warps store dS(j) only after
    the previous dQ product has read dS(j-1) (ds_free).  Checks: S and dP are read before the
    next product overwrites them, and dS is not overwritten while a dQ product reads it."""
    m.bar("s_ready")
    m.bar("dp_ready")
    m.bar("x_ready", 2)
    m.bar("dp_free", 2)
    m.bar("ds_ready", 2)
    m.bar("ds_free")
    m.bar("done")
    mma = [("mma", ["s_ready"]), ("mma", ["dp_ready"])]
    for j in range(n):
        mma.append(("wait", "x_ready", j))
        if j + 1 < n:
            mma.append(("mma", ["s_ready"]))
        mma.append(("wait", "dp_free", j))
        if j + 1 < n:
            mma.append(("mma", ["dp_ready"]))
        mma.append(("wait", "ds_ready", j))
        mma.append(("mma", ["ds_free"]))
    mma.append(("mma", ["done"]))

    def ew():
        e = []
        for j in range(n):
            e.append(("wait", "s_ready", j))
            e.append(("check", lambda mm, k=j + 1: mm.done["s_ready"] == k, "S overwritten before it was read"))
            e.append(("arrive", "x_ready"))
            e.append(("wait", "dp_ready", j))
            e.append(("check", lambda mm, k=j + 1: mm.done["dp_ready"] == k, "dP overwritten before it was read"))
            e.append(("arrive", "dp_free"))
            if j > 0:
                if not no_ds_free_wait:
                    e.append(("wait", "ds_free", j - 1))
                e.append(("check", lambda mm, k=j: mm.done["ds_free"] >= k, "dS stored while dQ read it"))
            e.append(("arrive", "ds_ready"))
        e.append(("wait", "done", 0))
        return e

    return {"mma": mma, "ew0": ew(), "ew1": ew()}


def bwd_dkdv_roles(m, n, no_dp_wait=False):
    """fa_bwd.cu's dK/dV kernel, one CTA over n query tiles; loads taken as ready; two
    elementwise groups stand for the eight warps, each staging its per-column vectors on
    its own (no barrier across warps).  dV += P^T dO_i once P^T is stored over S^T
    (x_ready), then S^T(i+1); dK += dS^T Q_i once dS^T is stored over dP^T (ds_ready), then
    dP^T(i+1).  Checks (with two commits the kernel does not need, to observe the products
    that read P^T and dS^T): a group reads S^T and dP^T of the current tile, and overwrites
    them only after the previous tile's dV and dK products have read them."""
    for b in ("s_ready", "dp_ready", "done", "dv_read", "dk_read"):
        m.bar(b)
    m.bar("x_ready", 2)
    m.bar("ds_ready", 2)
    mma = [("mma", ["s_ready"]), ("mma", ["dp_ready"])]
    for i in range(n):
        mma.append(("wait", "x_ready", i))
        mma.append(("mma", ["dv_read"]))
        if i + 1 < n:
            mma.append(("mma", ["s_ready"]))
        mma.append(("wait", "ds_ready", i))
        mma.append(("mma", ["dk_read"]))
        if i + 1 < n:
            mma.append(("mma", ["dp_ready"]))
    mma.append(("mma", ["done"]))

    def ew():
        e = []
        for i in range(n):
            e.append(("wait", "s_ready", i))
            e.append(("check", lambda mm, k=i + 1: mm.done["s_ready"] == k, "S^T not the current tile's"))
            e.append(("check", lambda mm, k=i: mm.done["dv_read"] >= k, "P^T stored while dV read the last one"))
            e.append(("arrive", "x_ready"))
            if not no_dp_wait:
                e.append(("wait", "dp_ready", i))
            e.append(("check", lambda mm, k=i + 1: mm.done["dp_ready"] == k, "dP^T not the current tile's"))
            e.append(("check", lambda mm, k=i: mm.done["dk_read"] >= k, "dS^T stored while dK read the last one"))
            e.append(("arrive", "ds_ready"))
        e.append(("wait", "done", 0))
        return e

    return {"mma": mma, "ew0": ew(), "ew1": ew()}


@pytest.mark.parametrize("n", [1, 2, 3, 5, 9])
def test_bwd_dq_protocol(n):
    for seed in range(150):
        m = Model(seed)
        res = m.run(bwd_dq_roles(m, n))
        assert res == "ok", (n, seed, res)


@pytest.mark.parametrize("n", [1, 2, 3, 5, 9])
def test_bwd_dkdv_protocol(n):
    for seed in range(150):
        m = Model(seed)
        res = m.run(bwd_dkdv_roles(m, n))
        assert res == "ok", (n, seed, res)


def test_bwd_dq_planted_missing_ds_free_fails():
    bad = 0
    for seed in range(200):
        m = Model(seed)
        bad += m.run(bwd_dq_roles(m, 4, no_ds_free_wait=True)).startswith("hazard")
    assert bad > 0


def test_bwd_dkdv_planted_missing_dp_wait_fails():
    bad = 0
    for seed in range(200):
        m = Model(seed)
        bad += m.run(bwd_dkdv_roles(m, 4, no_dp_wait=True)) != "ok"
    assert bad > 0
