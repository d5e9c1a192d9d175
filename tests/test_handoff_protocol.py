"""The dense kernel's named-barrier hand-offs, checked over every interleaving.

Hardware named barriers (`bar.sync` / `bar.arrive`) count arrivals, not who
arrives, and `bar.sync` has no timeout: if one warp arrives twice before its
partner arrives once, the generation completes with the wrong pair and the
partner then waits forever.  The MMA warps of fa_fwd_tiled_kernel hand work
over on such barriers:

  barrier 1 + t  scheduler -> issuer: groups 0 and 1 (Q.K^T of slot t) released
  barrier 3 + t  issuer -> scheduler: a group of slot t issued (back-pressure)
  barrier 5 + t  "P ready" of slot t: its four softmax warps, the scheduler
                 (the group's copies landed) and the issuer (192 threads)

This test writes down each role's sequence of barrier operations as the
kernel's loops produce them for slot tile counts (n0, n1), and explores all
interleavings: no state may deadlock, no warp may arrive twice in one
generation, and no arrival may be left over at the end.  The four softmax
warps of a slot act identically and are one agent of weight 4.

The rule that keeps it sound: a group past its slot's last tile (no P.V,
hence no Q.K^T) neither arrives on barrier 3 + t nor is waited for there.
The planted variant without that rule (every group arrives, the scheduler
waits for every group) must fail for every n0 != n1, which shows that the
check sees the hazard.  (Host-side model: it reads no file and runs no kernel.)
"""
import pytest

PREADY = 5
# expected arrivals per generation, in warps
EXPECT = {1: 2, 2: 2, 3: 2, 4: 2, 5: 6, 6: 6}


def role_programs(n0, n1, skip_empty=True):
    """Barrier programs of (scheduler, issuer, softmax slot 0, softmax slot 1)."""
    nt = (n0, n1)
    nmax = max(n0, n1)
    ngroups = 2 + 2 * nmax if nmax > 0 else 0

    def group(g):
        t = g if g < 2 else (g - 2) & 1
        jpv = -1 if g < 2 else (g - 2) >> 1
        return t, jpv, (0 <= jpv < nt[t]), (jpv + 1 < nt[t])

    sched = []
    for g in range(ngroups):
        t, jpv, pv_valid, _ = group(g)
        if g >= 2 and (not skip_empty or g < 4 or jpv <= nt[t]):
            sched.append(("sync", 3 + (g & 1)))       # issuer finished group g - 2
        if g < 2:
            sched.append(("arrive", 1 + g))
        elif pv_valid:
            sched.append(("arrive", PREADY + t))
    if skip_empty:
        if nmax > 0 and n0 == nmax:
            sched.append(("sync", 3))
        if nmax > 0 and n1 == nmax:
            sched.append(("sync", 4))
    elif ngroups:
        sched += [("sync", 3 + (ngroups & 1)), ("sync", 3 + ((ngroups - 1) & 1))]

    issuer = []
    for g in range(ngroups):
        t, jpv, pv_valid, qk_valid = group(g)
        if skip_empty and jpv >= 0 and not pv_valid:
            continue
        if jpv < 0:
            issuer.append(("sync", 1 + t))
        elif pv_valid:
            issuer.append(("sync", PREADY + t))
        if qk_valid:
            issuer.append(("s_ready", (t, jpv + 1)))   # commit of S_t for tile jpv + 1
        issuer.append(("arrive", 3 + t))

    softmax = []
    for t in range(2):
        prog = []
        for j in range(nt[t]):
            prog += [("wait", (t, j)), ("arrive", PREADY + t)]
        softmax.append(prog)
    return [sched, issuer] + softmax


def explore(progs, weights=(1, 1, 4, 4)):
    """Depth-first search of all interleavings; returns the first violation or None."""
    na = len(progs)
    bars = sorted(EXPECT)
    start = (tuple([0] * na), tuple([0] * na), tuple((0, frozenset()) for _ in bars), frozenset())
    seen, stack = set(), [start]
    while stack:
        state = stack.pop()
        if state in seen:
            continue
        seen.add(state)
        pcs, blocked, bstate, events = state
        moved = False
        for a in range(na):
            if blocked[a] or pcs[a] >= len(progs[a]):
                continue
            op, arg = progs[a][pcs[a]]
            if op == "wait" and arg not in events:
                continue
            moved = True
            pcs2, blk2, bs2, ev2 = list(pcs), list(blocked), list(bstate), events
            pcs2[a] += 1
            if op == "s_ready":
                ev2 = events | {arg}
            elif op in ("arrive", "sync"):
                i = bars.index(arg)
                count, who = bs2[i]
                if a in who:
                    return f"role {a} arrives twice in one generation of barrier {arg}"
                count += weights[a]
                who = who | {a}
                if op == "sync":
                    blk2[a] = arg
                if count == EXPECT[arg]:
                    blk2 = [0 if b == arg else b for b in blk2]
                    count, who = 0, frozenset()
                elif count > EXPECT[arg]:
                    return f"barrier {arg} over-subscribed"
                bs2[i] = (count, who)
            stack.append((tuple(pcs2), tuple(blk2), tuple(bs2), ev2))
        if not moved:
            if any(blocked[a] or pcs[a] < len(progs[a]) for a in range(na)):
                return f"deadlock: positions {pcs}, waiting on {blocked}"
            if any(c for c, _ in bstate):
                return "arrivals left over at exit"
    return None


@pytest.mark.parametrize("n0", range(7))
def test_handoffs_never_hang(n0):
    for n1 in range(7):
        assert explore(role_programs(n0, n1)) is None, (n0, n1)


def test_planted_rule_without_the_empty_group_skip_hangs():
    bad = [(n0, n1) for n0 in range(4) for n1 in range(4)
           if explore(role_programs(n0, n1, skip_empty=False)) is not None]
    assert bad == [(n0, n1) for n0 in range(4) for n1 in range(4) if n0 != n1]
