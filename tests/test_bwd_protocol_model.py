"""The backward kernels' mbarrier hand-offs (attention_forward_fa_gb300/csrc/
fa_bwd.cuh), checked over every interleaving before any GPU run.

Roles of one CTA (the dK / dV and dQ kernels share the protocol): the TMA
producer, the MMA issuer, and the four elementwise warps (one agent: they
arrive on p_ready once each, count 4).  Asynchronous completions are agents
too: each TMA copy lands at any time after it was issued; tcgen05 commits
complete in issue order, each after every MMA issued before it.

mbarrier waits are parity waits: try_wait.parity(P) passes once the barrier
has completed a phase of parity P, i.e. while (completed phases) & 1 != P.
Besides deadlock, the check looks for the hazard that parity waits cannot
see: a barrier running two phases ahead of a waiter (the waiter would then
block on a later phase).  It also checks that a ring stage is reloaded only
after the products that read it completed, and that S of a step is
overwritten only after the elementwise warps read it, and that the products
read P / dS only after the elementwise warps wrote them.
"""
import pytest


def programs(nsteps, planted=None):
    """Each role's operations as the kernels order them; ``planted`` names a
    deliberate mistake (for the test that the check sees it)."""
    prod = [("issue_tma", "res", None)]
    for n in range(nsteps):
        s = n & 1
        if n >= 2 and planted != "no_empty_wait":
            prod.append(("wait", f"empty{s}", (n >> 1) - 1, f"reload stage {s} for step {n}"))
        elif n >= 2:
            prod.append(("check_reload", n))
        prod.append(("issue_tma", f"full{s}", n))
    mma = [("wait", "res", 0, None)]
    for n in range(nsteps):
        s = n & 1
        step = [("wait", f"full{s}", n >> 1, None),
                ("read_stage", s, n),
                ("issue_mma_commit", "s_ready", n),          # S^T / dP^T products, then commit
                ("wait", "p_ready", n, None),
                ("issue_mma_commit", f"empty{s}", n)]        # dV / dK (or dQ) products, then commit
        if planted == "s_before_p":
            step[2], step[3] = step[3], step[2]
            step[2] = ("wait", "p_ready", n - 1, None) if n else ("nop",)
            step[3] = ("issue_mma_commit", "s_ready", n)
        mma += step
    mma.append(("issue_mma_commit", "acc", None))
    elem = []
    for n in range(nsteps):
        if planted == "elem_no_wait":
            elem += [("read_s", n), ("arrive", "p_ready", 4)]
        else:
            elem += [("wait", "s_ready", n, None), ("read_s", n), ("arrive", "p_ready", 4)]
    if nsteps:
        elem.append(("wait", "acc", 0, None))
    return prod, mma, elem


COUNTS = {"res": 1, "full0": 1, "full1": 1, "empty0": 1, "empty1": 1, "s_ready": 1, "p_ready": 4,
          "acc": 1}


def explore(nsteps, planted=None):
    prod, mma, elem = programs(nsteps, planted)
    progs = [prod, mma, elem]
    bars0 = tuple((0, 0) for _ in COUNTS)          # (completed phases, pending arrivals)
    names = list(COUNTS)
    # state: pcs, barriers, in-flight TMA copies (set), MMA commit queue (tuple, in order),
    # stage reads done (set of steps), S reads done (set)
    start = ((0, 0, 0), bars0, frozenset(), (), frozenset(), frozenset())
    seen, stack = set(), [start]
    while stack:
        st = stack.pop()
        if st in seen:
            continue
        seen.add(st)
        pcs, bars, tma, queue, sread, sdone = st
        moved = False

        def arrive(bars, name, k=1):
            i = names.index(name)
            done, pend = bars[i]
            pend += k
            if pend == COUNTS[name]:
                done, pend = done + 1, 0
            elif pend > COUNTS[name]:
                raise AssertionError(f"{name} over-arrived")
            return bars[:i] + ((done, pend),) + bars[i + 1:]

        for a in range(3):
            if pcs[a] >= len(progs[a]):
                continue
            op = progs[a][pcs[a]]
            nb, ntma, nq, nsr, nsd = bars, tma, queue, sread, sdone
            if op[0] == "wait":
                _, name, phase, what = op
                done = bars[names.index(name)][0]
                assert done <= phase + 1, f"{name} ran two phases ahead of a waiter (phase {phase})"
                if done <= phase:           # parity wait passes once phase `phase` completed
                    continue
                if what and what.startswith("reload stage"):
                    n = int(what.split()[-1])
                    assert (n - 2) in sread, "stage reloaded before the products that read it"
            elif op[0] == "nop":
                pass
            elif op[0] == "check_reload":
                assert (op[1] - 2) in sread, "stage reloaded before the products that read it"
            elif op[0] == "issue_tma":
                ntma = tma | {op[1:]}
            elif op[0] == "read_stage":
                nsr = sread | {op[2]}
            elif op[0] == "issue_mma_commit":
                if op[1] == "s_ready" and op[2] >= 1:
                    assert (op[2] - 1) in sdone, "S overwritten before the elementwise warps read it"
                if op[1].startswith("empty"):   # the products that read P / dS of step op[2]
                    assert bars[names.index("p_ready")][0] > op[2], "P / dS read before they were written"
                nq = queue + (op[1],)
            elif op[0] == "read_s":
                assert op[1] < 0 or bars[names.index("s_ready")][0] > op[1], "S read before it was ready"
                nsd = sdone | {op[1]}
            elif op[0] == "arrive":
                nb = arrive(bars, op[1], op[2])
            moved = True
            npcs = list(pcs)
            npcs[a] += 1
            stack.append((tuple(npcs), nb, ntma, nq, nsr, nsd))
        for cp in tma:                       # a copy lands
            moved = True
            stack.append((pcs, arrive(bars, cp[0]), tma - {cp}, queue, sread, sdone))
        if queue:                            # the oldest commit completes
            moved = True
            stack.append((pcs, arrive(bars, queue[0]), tma, queue[1:], sread, sdone))
        if not moved:
            assert all(pcs[a] >= len(progs[a]) for a in range(3)), f"deadlock at {pcs}"
    return len(seen)


@pytest.mark.parametrize("nsteps", [0, 1, 2, 3, 4, 5])
def test_backward_handoffs_never_hang_or_alias(nsteps):
    assert explore(nsteps) > 0


@pytest.mark.parametrize("planted", ["no_empty_wait", "s_before_p", "elem_no_wait"])
def test_planted_mistakes_are_seen(planted):
    with pytest.raises(AssertionError):
        explore(4, planted)
