"""The top-k kernel's ring hand-offs, with the producers' copy window, checked
over every interleaving.

fa_mla_topk_kernel gathers each 64-key tile into one of two ring stages, as
two regions with their own full / empty mbarriers: X (the boxes read by the
X steps of Q.K^T only) and V (the boxes read by the V steps of Q.K^T and by
P.V).  Region r = 2j + e is tile j's X (e = 0) or V (e = 1) region.  The
producer warps issue region r's copies once its empty barrier allows (or,
on a stage's first use, once the Q staging that held the stage is consumed),
and keep `depth` regions in flight: after issuing region r they wait for the
copies of region r - depth + 1 alone and arrive on its full barrier.  The MMA
warp issues, per tile j, the X steps of S_j, P.V of tile j - 1 and the V
steps of S_j; its commits release S to the softmax, X once Q.K^T of the tile
is complete and V once its P.V is.  The softmax warps hand S back as soon as
they hold it, and P once written.

This test writes down each role's sequence of barrier operations for a tile
count nt and explores all interleavings: every state must be able to move
until all roles finish, and no wait may pass while its barrier could be two
phases ahead (an mbarrier wait tells phases apart by parity only).  The
producers (three warps acting alike) and the softmax warps (four) are one
agent each; commits arrive when the MMA warp issues them, since an MMA, once
issued, waits on nothing.  Windows of one, two and three regions are sound;
four must deadlock from the third tile on (X of tile j waits for Q.K^T of
tile j - 2, which needs V of tile j - 2, three regions back), which shows
that the check sees the hazard.  Each tile has one P.V pass here; the
residual pass of a short or lazily rescaled tile adds one more P-ready /
P.V-done pair, which the softmax and the MMA warp count alike and which
touches no ring barrier.  (Host-side model: it reads no file and runs no
kernel.)
"""
import pytest

NS = 2   # ring stages


def programs(nt, depth):
    """Barrier programs of (producers, MMA warp, softmax) for nt tiles."""
    full = lambda r: ("FULL_V" if r & 1 else "FULL_X", (r >> 1) % NS)   # noqa: E731
    prod = []
    for r in range(2 * nt):
        j, e = r >> 1, r & 1
        s, use = j % NS, j // NS
        if use == 0:
            if e == 0:
                prod.append(("wait", ("QDONE", 0), 0))
        else:
            prod.append(("wait", ("EMPTY_V" if e else "EMPTY_X", s), use - 1))
        # copies of region r issued; region r - depth + 1 landed
        if r - depth + 1 >= 0:
            prod.append(("arrive", full(r - depth + 1)))
    for r in range(max(0, 2 * nt - depth + 1), 2 * nt):
        prod.append(("arrive", full(r)))

    mma = [("wait", ("QDONE", 0), 0)]
    for j in range(nt + 1):
        s, use = j % NS, j // NS
        if j < nt:
            if j > 0:
                mma.append(("wait", ("SFREE", 0), j - 1))
            mma.append(("wait", ("FULL_X", s), use))
        if j > 0:
            sp = (j - 1) % NS
            mma.append(("wait", ("PREADY", 0), j - 1))
            mma.append(("arrive", ("PVDONE", 0)))
            mma.append(("arrive", ("EMPTY_V", sp)))
        if j < nt:
            mma.append(("wait", ("FULL_V", s), use))
            mma.append(("arrive", ("SFULL", 0)))
            mma.append(("arrive", ("EMPTY_X", s)))

    soft = [("wait", ("QFULL", 0), 0), ("arrive", ("QDONE", 0))]
    for j in range(nt):
        soft.append(("wait", ("SFULL", 0), j))
        soft.append(("arrive", ("SFREE", 0)))
        if j > 0:
            soft.append(("wait", ("PVDONE", 0), j - 1))
        soft.append(("arrive", ("PREADY", 0)))
    if nt > 0:
        soft.append(("wait", ("PVDONE", 0), nt - 1))
    return [prod, mma, soft]


def explore(progs):
    """All interleavings.  Returns (deadlock state or None, parity hazards)."""
    bars = sorted({op[1] for p in progs for op in p})
    index = {b: i for i, b in enumerate(bars)}
    start = tuple([0] * len(progs)) + tuple(1 if b == ("QFULL", 0) else 0 for b in bars)
    n = len(progs)
    seen = {start}
    stack = [start]
    hazards = set()
    while stack:
        st = stack.pop()
        pcs, done = st[:n], st[n:]
        if all(pcs[a] == len(progs[a]) for a in range(n)):
            continue
        moved = False
        for a in range(n):
            if pcs[a] == len(progs[a]):
                continue
            op = progs[a][pcs[a]]
            c = list(done)
            if op[0] == "wait":
                k = done[index[op[1]]]
                if k < op[2] + 1:
                    continue           # phase op[2] not complete yet
                if k > op[2] + 1:
                    hazards.add((a, op))   # two phases ahead: parity would be wrong
            else:
                c[index[op[1]]] += 1
            p2 = list(pcs)
            p2[a] += 1
            nxt = tuple(p2) + tuple(c)
            moved = True
            if nxt not in seen:
                seen.add(nxt)
                stack.append(nxt)
        if not moved:
            return st, hazards
    return None, hazards


@pytest.mark.parametrize("depth", [1, 2, 3])
@pytest.mark.parametrize("nt", [1, 2, 3, 4, 5, 6])
def test_copy_windows_up_to_three_regions_are_sound(nt, depth):
    dead, hazards = explore(programs(nt, depth))
    assert dead is None, f"deadlock at {dead}"
    assert not hazards, hazards


@pytest.mark.parametrize("nt", [3, 4, 5])
def test_a_four_region_window_deadlocks(nt):
    dead, _ = explore(programs(nt, 4))
    assert dead is not None


@pytest.mark.parametrize("nt", [1, 2])
def test_a_four_region_window_is_harmless_on_short_lists(nt):
    # with at most two tiles no empty barrier is waited on (every stage's first use)
    dead, hazards = explore(programs(nt, 4))
    assert dead is None and not hazards
