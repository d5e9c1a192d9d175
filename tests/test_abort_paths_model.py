"""The kernels' failure paths, checked over every interleaving on the CPU.

Every mbarrier wait in the kernels is bounded: once its limit passes, or once
another thread of the CTA gave up (the CTA's abort flag), the waiting role
stops waiting and takes its failure path.  Hardware named barriers
(`bar.sync`) and the final `__syncthreads` have no limit, so a failure path
that leaves one of them short of arrivals, or completes a generation with the
wrong set of warps, would hang the GPU instead of reporting
FA_ERR_DEVICE_TIMEOUT.  This model lets any role give up at any bounded wait
whose event has not happened yet, at any moment, and checks:

  * no interleaving ends with a role stuck at a named barrier or the CTA
    barrier (every `bar.sync` generation still completes);
  * no named-barrier generation receives two arrivals of one role, or more
    arrivals than it expects, and none is left half-full at exit;
  * when the CTA's barrier releases the teardown, no TMA copy is still in
    flight and every tensor-core commit has completed (shared memory and
    TMEM are released only after their last writer);
  * before any role gave up, no parity wait passes on a phase other than the
    one it waits for (a barrier two phases ahead of its waiter).

Drain waits (the teardown's waits that ignore the abort flag, bounded by at
least 100 ms) block until their event; the model lets one end by its limit
only when nothing else in the CTA can move, i.e. when the event can never
happen, and counts that.

The roles' programs are written down from the kernels' loops:
attention_forward_fa_gb300/csrc/fa_tiled.cuh (the dense forward: TMA producer,
V converter, MMA scheduler, MMA issuer, the softmax warps of two query
tiles, which also write their tile's epilogue) and csrc/fa_bwd.cuh (the
backward's dK/dV kernel: producer, MMA issuer, four elementwise warps).  Planted mistakes show that each property is
seen.  Host-side model: it reads no file and runs no kernel.
"""
import pytest


# ------------------------------------------------------------------ checker

class Violation(AssertionError):
    pass


def explore(roles, mbar_counts, nbar_expect, limit=3_000_000):
    """roles: list of (name, weight, {program name: [ops]}); every role starts
    in its program "main".  Returns (states seen, drains that ended by their
    limit).  Raises Violation on the first property that fails."""
    names = [r[0] for r in roles]
    weights = [r[1] for r in roles]
    progs = [r[2] for r in roles]
    mbars = sorted(mbar_counts)
    nbars = sorted(nbar_expect)
    na = len(roles)

    def passes(c, k):
        # try_wait.parity(k & 1) passes while the current phase's parity differs
        return (c & 1) != (k & 1)

    start = (tuple(["main"] * na), tuple([0] * na), tuple([None] * na),
             tuple((0, 0) for _ in mbars), tuple((0, frozenset()) for _ in nbars),
             (), (), False, frozenset(), 0)
    seen = set()
    stack = [start]
    expired_max = 0
    while stack:
        st = stack.pop()
        if st in seen:
            continue
        if len(seen) > limit:
            raise RuntimeError("state space too large")
        seen.add(st)
        pn, pcs, blocked, mb, nb, tma, queue, abort, at_sync, expired = st
        expired_max = max(expired_max, expired)

        def mb_arrive(mb, bar, k=1):
            i = mbars.index(bar)
            c, pend = mb[i]
            pend += k
            if pend == mbar_counts[bar]:
                c, pend = c + 1, 0
            elif pend > mbar_counts[bar]:
                raise Violation(f"mbarrier {bar} over-arrived")
            return mb[:i] + ((c, pend),) + mb[i + 1:]

        succ = []
        drains = []
        for a in range(na):
            if blocked[a] is not None:
                continue
            prog = progs[a][pn[a]]
            if pcs[a] >= len(prog):
                continue
            op = prog[pcs[a]]
            kind = op[0]

            def nxt(**chg):
                d = dict(pn=pn, pcs=pcs, blocked=blocked, mb=mb, nb=nb, tma=tma, queue=queue,
                         abort=abort, at_sync=at_sync, expired=expired)
                npcs = list(pcs)
                npcs[a] += 1
                d["pcs"] = tuple(npcs)
                d.update(chg)
                return (d["pn"], d["pcs"], d["blocked"], d["mb"], d["nb"], d["tma"], d["queue"],
                        d["abort"], d["at_sync"], d["expired"])

            if kind in ("tma", "commit"):
                # invisible to the other roles (they see a copy only when it
                # lands and a commit only when it completes, both separate
                # moves): taken together with every such step that follows
                ntma, nq, k = tma, queue, pcs[a]
                while k < len(prog) and prog[k][0] in ("tma", "commit"):
                    if prog[k][0] == "tma":
                        ntma = tuple(sorted(ntma + (prog[k][1],)))
                    else:
                        nq = nq + (prog[k][1],)
                    k += 1
                npcs = list(pcs)
                npcs[a] = k
                succ.append(nxt(tma=ntma, queue=nq, pcs=tuple(npcs)))
            elif kind == "arrive":
                succ.append(nxt(mb=mb_arrive(mb, op[1], op[2] if len(op) > 2 else 1)))
            elif kind == "set_abort":
                succ.append(nxt(abort=True))
            elif kind == "ifabort":
                if abort:
                    npn = list(pn)
                    npn[a] = op[1]
                    npcs = list(pcs)
                    npcs[a] = 0
                    succ.append(nxt(pn=tuple(npn), pcs=tuple(npcs)))
                else:
                    succ.append(nxt())
            elif kind == "ext_wait":
                # an event outside the model: it may come, or the wait may give up
                succ.append(nxt())
                npn = list(pn)
                npn[a] = op[1]
                npcs = list(pcs)
                npcs[a] = 0
                succ.append(nxt(pn=tuple(npn), pcs=tuple(npcs), abort=True))
            elif kind in ("bwait", "drain"):
                bar, k = op[1], op[2]
                c = mb[mbars.index(bar)][0]
                if passes(c, k):
                    if not abort and c != k + 1:
                        raise Violation(f"{names[a]}: wait on {bar} passed on phase {c - 1}, "
                                        f"not {k} (barrier two phases ahead)")
                    succ.append(nxt())
                elif kind == "bwait":
                    # give up: the failure path, and the CTA's abort flag
                    npn = list(pn)
                    npn[a] = op[3]
                    npcs = list(pcs)
                    npcs[a] = 0
                    succ.append(nxt(pn=tuple(npn), pcs=tuple(npcs), abort=True))
                else:
                    drains.append(a)
            elif kind in ("nbsync", "nbarrive"):
                bid = op[1]
                i = nbars.index(bid)
                cnt, who = nb[i]
                if a in who:
                    raise Violation(f"{names[a]} arrives twice in one generation of named "
                                    f"barrier {bid}")
                cnt += weights[a]
                who = who | {a}
                nblk = list(blocked)
                if kind == "nbsync":
                    nblk[a] = bid
                if cnt == nbar_expect[bid]:
                    nblk = [None if b == bid else b for b in nblk]
                    cnt, who = 0, frozenset()
                elif cnt > nbar_expect[bid]:
                    raise Violation(f"named barrier {bid} over-subscribed")
                nnb = nb[:i] + ((cnt, who),) + nb[i + 1:]
                succ.append(nxt(nb=nnb, blocked=tuple(nblk)))
            elif kind == "syncall":
                nblk = list(blocked)
                nblk[a] = "syncall"
                ats = at_sync | {a}
                if len(ats) == na:
                    if tma:
                        raise Violation(f"teardown with TMA copies in flight: {tma}")
                    if queue:
                        raise Violation(f"teardown with tensor-core commits pending: {queue}")
                    if any(cnt for cnt, _ in nb):
                        raise Violation("named-barrier arrivals left over at exit")
                    nblk = [None] * na
                succ.append(nxt(blocked=tuple(nblk), at_sync=ats))
            else:
                raise ValueError(op)
        for bar in sorted(set(tma)):          # a copy lands
            lst = list(tma)
            lst.remove(bar)
            succ.append((pn, pcs, blocked, mb_arrive(mb, bar), nb, tuple(lst), queue, abort,
                         at_sync, expired))
        if queue:                             # the oldest commit completes
            succ.append((pn, pcs, blocked, mb_arrive(mb, queue[0]), nb, tma, queue[1:], abort,
                         at_sync, expired))
        if not succ and drains:
            # nothing else can move: a drain ends by its limit
            for a in drains:
                npcs = list(pcs)
                npcs[a] += 1
                succ.append((pn, tuple(npcs), blocked, mb, nb, tma, queue, abort, at_sync,
                             expired + 1))
        if not succ:
            done = all(pcs[a] >= len(progs[a][pn[a]]) and blocked[a] is None for a in range(na))
            if not done:
                where = {names[a]: (pn[a], pcs[a], blocked[a]) for a in range(na)
                         if blocked[a] is not None or pcs[a] < len(progs[a][pn[a]])}
                raise Violation(f"hang: {where}")
        stack.extend(succ)
    return len(seen), expired_max


# ------------------------------------------------------------------ dense forward

PREADY = 5


def _forward_plan(n0, n1, NS):
    """The dense kernel's load order and MMA groups for one CTA whose slots have
    n0 and n1 KV tiles (event_at / num_events and the scheduler's bookkeeping
    of fa_tiled.cuh)."""
    nt = (n0, n1)
    nmax = max(n0, n1)
    shared = n0 >= 1 and n0 <= n1
    loads = []
    for e in range(2 + 4 * nmax if nmax > 0 else 0):
        if e < 2:
            pv, t, j = False, e, 0
        else:
            r, jj = (e - 2) & 3, (e - 2) >> 2
            pv, t = (r & 1) == 0, r >> 1
            j = jj if pv else jj + 1
        if j < nt[t] and ((t == 0 or j >= n0) if shared else True):
            L = len(loads)
            loads.append((L, L % NS, L // NS))
    groups = []
    ld = 0
    for g in range(2 + 2 * nmax if nmax > 0 else 0):
        t = g if g < 2 else (g - 2) & 1
        jpv = -1 if g < 2 else (g - 2) >> 1
        jqk = 0 if g < 2 else jpv + 1
        ntt = nt[t]
        pv_valid = 0 <= jpv < ntt
        qk_valid = jqk < ntt
        pv_load = pv_valid and (not shared or t == 0 or jpv >= n0)
        qk_load = qk_valid and (not shared or t == 0 or jqk >= n0)
        if shared:
            lpv, lqk = 2 * jpv + 1, 2 * jqk
        else:
            lpv, lqk = ld, ld + (1 if pv_load else 0)
            ld += (1 if pv_load else 0) + (1 if qk_load else 0)
        groups.append((g, t, jpv, jqk, ntt, pv_valid, qk_valid, pv_load, qk_load, lpv, lqk))
    return nt, nmax, shared, loads, groups


def _scheduler_ops(nt, nmax, n0, n1, groups, NS, waits):
    """Warp 14: per group, the issuer's "group issued" barrier, the bounded
    waits for the group's copies (``waits``: "mbar" = real READY / QFULL waits,
    "ext" = an event outside the model, which may come or not), the release."""
    ops = []
    for g, t, jpv, jqk, ntt, pv_valid, qk_valid, pv_load, qk_load, lpv, lqk in groups:
        if g >= 2 and (g < 4 or jpv <= ntt):
            ops.append(("nbsync", 3 + (g & 1)))
        w = []
        if pv_load:
            w.append((f"ready{lpv % NS}", lpv // NS))
        if qk_load:
            w.append((f"ready{lqk % NS}", lqk // NS))
        if qk_valid and jqk == 0:
            w.append((f"qfull{t}", 0))
        for bar, k in w:
            ops.append(("bwait", bar, k) if waits == "mbar" else ("ext_wait",))
        if g < 2:
            ops.append(("nbarrive", 1 + g))
        elif pv_valid:
            ops.append(("nbarrive", PREADY + t))
    if nmax > 0 and n0 == nmax:
        ops.append(("nbsync", 3))
    if nmax > 0 and n1 == nmax:
        ops.append(("nbsync", 4))
    return ops + [("syncall",)]


def _with_giveups(ops, planted=None):
    """The scheduler's program and its failure paths: after a wait gave up it
    skips every later wait but still releases every group (the issuer then
    runs on stale operands; nothing waits on the results)."""
    prog = {"main": []}
    for i, op in enumerate(ops):
        if op[0] in ("bwait", "ext_wait"):
            alt = f"aborted{i}"
            rest = [o for o in ops[i + 1:] if o[0] not in ("bwait", "ext_wait")]
            if planted == "scheduler_stops":
                rest = [o for o in rest if o[0] == "syncall"]
            prog[alt] = rest
            prog["main"].append(op + (alt,))
        else:
            prog["main"].append(op)
    return prog


def forward_handoff_roles(n0, n1, NS=2, planted=None):
    """Model A: the named-barrier hand-offs of fa_tiled.cuh.  The MMA scheduler
    (its waits for TMA copies and the V converter are events outside this
    model: each may come or give up at any time), the MMA issuer, and the
    softmax warps of both slots (one agent of weight 4 each)."""
    nt, nmax, shared, loads, groups = _forward_plan(n0, n1, NS)
    sched = _with_giveups(_scheduler_ops(nt, nmax, n0, n1, groups, NS, "ext"), planted)
    iss = {"main": []}
    for g, t, jpv, jqk, ntt, pv_valid, qk_valid, pv_load, qk_load, lpv, lqk in groups:
        if jpv >= 0 and not pv_valid:
            continue
        iss["main"].append(("nbsync", 1 + t) if jpv < 0 else ("nbsync", PREADY + t))
        if pv_valid and jpv == ntt - 1:
            iss["main"].append(("commit", f"oready{t}"))   # the slot's last P.V
        if qk_valid:
            iss["main"].append(("commit", f"sfull{t}"))
        iss["main"].append(("nbarrive", 3 + t))
    if n0 + n1 > 0:
        iss["main"] += [("commit", "drain"), ("drain", "drain", 0)]
    iss["main"].append(("syncall",))

    def softmax(t):
        # after its last tile the slot's warps write its epilogue once its
        # last P.V has completed (a bounded wait; on a give-up the slot's
        # warps agree to skip the writes); the warps of one slot move as one
        # agent here, so their own staging barrier is not modelled
        pr = {"main": [], "epi_skip": [("syncall",)]}
        tail = ([("bwait", f"oready{t}", 0, "epi_skip")] if nt[t] > 0 else []) + [("syncall",)]
        for j in range(nt[t]):
            alt = f"dead{j}"
            dead = []
            for j2 in range(j, nt[t]):
                # every arrival after giving up, the given-up tile's included,
                # is paced by the issuer's S commit of that tile (planted: no
                # pacing, or none for the tile it gave up on)
                paced = planted != "softmax_unpaced" and \
                    not (planted == "softmax_unpaced_at_giveup" and j2 == j)
                if paced:
                    dead.append(("drain", f"sfull{t}", j2))
                dead.append(("nbarrive", PREADY + t))
            pr[alt] = dead + [("syncall",)]   # a warp that gave up skips the epilogue
            pr["main"] += [("bwait", f"sfull{t}", j, alt), ("nbarrive", PREADY + t)]
        pr["main"] += tail
        return pr

    roles = [("scheduler", 1, sched), ("issuer", 1, iss), ("softmax0", 4, softmax(0)),
             ("softmax1", 4, softmax(1))]
    mcounts = {"sfull0": 1, "sfull1": 1, "oready0": 1, "oready1": 1, "drain": 1}
    return roles, mcounts, {1: 2, 2: 2, 3: 2, 4: 2, 5: 6, 6: 6}


def forward_ring_roles(n0, n1, NS=2, planted=None):
    """Model B: the ring of fa_tiled.cuh and the teardown.  The TMA producer,
    the V converter, and the MMA side as one consumer: the scheduler's waits
    for each group's copies, then the issuer's commits that release the
    group's stages."""
    nt, nmax, shared, loads, groups = _forward_plan(n0, n1, NS)

    def drains(issued):
        ops = [("drain", f"full{L % NS}", L // NS) for L in range(max(0, issued - NS), issued)]
        return ops + [("drain", f"qfull{t}", 0) for t in range(2) if nt[t] > 0]

    prod = {"main": [("tma", f"qfull{t}") for t in range(2) if nt[t] > 0]}
    for L, s, f in loads:
        if L >= 1:
            alt = f"break{L}"
            prod[alt] = (drains(L) if planted != "producer_no_drain" else []) + [("syncall",)]
            prod["main"].append(("bwait", f"empty{s}", f - 1, alt))
            if f > 0 and planted != "producer_reuses_unlanded":
                # the stage's previous copy has landed
                prod["main"].append(("bwait", f"full{s}", f - 1, alt))
        prod["main"].append(("tma", f"full{s}"))
    if planted != "producer_no_drain":
        prod["main"] += drains(len(loads))
    prod["main"].append(("syncall",))

    conv = {"main": []}
    for L, s, f in loads:
        alt = f"dead{L}"
        conv[alt] = [("arrive", f"ready{s2}") for _, s2, _ in loads[L:]] + [("syncall",)]
        conv["main"] += [("bwait", f"full{s}", f, alt), ("arrive", f"ready{s}")]
    conv["main"] += [("syncall",)]

    cons_ops = []
    for g, t, jpv, jqk, ntt, pv_valid, qk_valid, pv_load, qk_load, lpv, lqk in groups:
        if pv_load:
            cons_ops.append(("bwait", f"ready{lpv % NS}", lpv // NS))
        if qk_load:
            cons_ops.append(("bwait", f"ready{lqk % NS}", lqk // NS))
        if qk_valid and jqk == 0:
            cons_ops.append(("bwait", f"qfull{t}", 0))
        if pv_valid and (not shared or t == 1):
            cons_ops.append(("commit", f"empty{lpv % NS}"))
        if qk_valid and (not shared or t == 1):
            cons_ops.append(("commit", f"empty{lqk % NS}"))
    if n0 + n1 > 0:
        cons_ops += [("commit", "drain"), ("drain", "drain", 0)]
    cons_ops.append(("syncall",))
    cons = _with_giveups(cons_ops)

    mcounts = {"drain": 1}
    for s in range(NS):
        mcounts.update({f"full{s}": 1, f"empty{s}": 1, f"ready{s}": 1})
    for t in range(2):
        mcounts[f"qfull{t}"] = 1
    return [("producer", 1, prod), ("converter", 1, conv), ("consumer", 1, cons)], mcounts, {}


FWD_CASES = [(n0, n1) for n0 in range(3) for n1 in range(3)]


@pytest.mark.parametrize("n0,n1", FWD_CASES)
def test_forward_handoffs_survive_every_failure_path(n0, n1):
    states, expired = explore(*forward_handoff_roles(n0, n1))
    assert states > 0
    assert expired == 0   # no drain waits out its limit: every event it waits for comes


@pytest.mark.parametrize("n0,n1", FWD_CASES + [(3, 3), (2, 3)])
def test_forward_ring_and_teardown_survive_every_failure_path(n0, n1):
    states, expired = explore(*forward_ring_roles(n0, n1))
    assert states > 0


@pytest.mark.parametrize("planted,model,n0,n1", [
    ("scheduler_stops", forward_handoff_roles, 1, 1),
    ("softmax_unpaced", forward_handoff_roles, 2, 2),
    ("softmax_unpaced_at_giveup", forward_handoff_roles, 2, 2),
    ("producer_reuses_unlanded", forward_ring_roles, 2, 2),
    ("producer_no_drain", forward_ring_roles, 1, 1),
])
def test_forward_planted_failure_path_mistakes_are_seen(planted, model, n0, n1):
    with pytest.raises(Violation):
        explore(*model(n0, n1, planted=planted))


# ------------------------------------------------------------------ backward (dK / dV kernel)

def backward_roles(nsteps, planted=None):
    """fa_bwd_dkdv_kernel's roles (fa_bwd.cuh): the TMA producer, the MMA
    issuer, and the four elementwise warps as two agents of two warps each
    (so that warps can take different paths: each agent arrives on p_ready
    with its two warps once per step, and all four warps meet at named
    barrier 1 once per step, before the step's S wait)."""
    def prod_drains(issued):
        ops = [("drain", "res", 0)]
        return ops + [("drain", f"full{i & 1}", i >> 1) for i in range(max(0, issued - 2), issued)]

    prod = {"main": []}
    if nsteps > 0:
        prod["main"].append(("tma", "res"))
        for n in range(nsteps):
            s = n & 1
            alt = f"break{n}"
            prod[alt] = (prod_drains(n) if planted != "producer_no_drain" else []) + [("syncall",)]
            prod["main"] += [("bwait", f"empty{s}", (n >> 1) - 1, alt), ("tma", f"full{s}")]
        if planted != "producer_no_drain":
            prod["main"] += prod_drains(nsteps)
    prod["main"].append(("syncall",))

    end = [("commit", "acc"), ("commit", "drain"), ("drain", "drain", 0), ("syncall",)]
    iss = {"main": [], "fail": [("set_abort",)] + end}
    if nsteps > 0:
        iss["main"].append(("bwait", "res", 0, "fail"))
        for n in range(nsteps):
            s = n & 1
            iss["main"] += [("bwait", f"full{s}", n >> 1, "fail"), ("commit", "s_ready"),
                            ("bwait", "p_ready", n, "fail"), ("commit", f"empty{s}")]
    iss["main"] += end

    def elem():
        pr = {"main": [], "epi_none": [("syncall",)]}
        epi = [("bwait", "acc", 0, "epi_none")] if nsteps > 0 else []
        for n in range(nsteps):
            alt = f"dead{n}"
            dead = [("arrive", "p_ready", 2)]
            for _ in range(n + 1, nsteps):
                if planted != "dead_skips_step_barrier":
                    dead.append(("nbsync", 1))
                dead.append(("arrive", "p_ready", 2))
            pr[alt] = dead + [("syncall",)]
            pr["main"] += [("nbsync", 1), ("bwait", "s_ready", n, alt), ("arrive", "p_ready", 2)]
        pr["main"] += epi + [("syncall",)]
        return pr

    roles = [("producer", 1, prod), ("issuer", 1, iss), ("elem01", 2, elem()), ("elem23", 2, elem())]
    mcounts = {"res": 1, "full0": 1, "full1": 1, "empty0": 1, "empty1": 1, "s_ready": 1,
               "p_ready": 4, "acc": 1, "drain": 1}
    return roles, mcounts, {1: 4}


@pytest.mark.parametrize("nsteps", [0, 1, 2, 3])
def test_backward_failure_paths_never_hang(nsteps):
    states, expired = explore(*backward_roles(nsteps))
    assert states > 0


@pytest.mark.parametrize("planted", ["dead_skips_step_barrier", "producer_no_drain"])
def test_backward_planted_failure_path_mistakes_are_seen(planted):
    with pytest.raises(Violation):
        explore(*backward_roles(3, planted=planted))
