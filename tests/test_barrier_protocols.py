"""Models of the mbarrier protocols of the tcgen05 attention kernels
(sparse_backward_gemm_gb300/csrc/attn.cu), checked on the CPU.

Each role of a kernel (TMA producer, MMA issuer, softmax groups, epilogue) is
written as its sequence of waits and arrivals; an event is (barrier, phase).
Two properties are checked for every sequence length:
  * no deadlock: run to quiescence, every role finishes;
  * no missed phase: every wait is a parity wait, so a wait for phase k of a
    barrier must never find phase k+1 already complete (the parity would read
    as "not yet" and the wait would run out).  With the waiting role frozen
    just before that wait and every other role run as far as it can, phase
    k+1 of that barrier must not complete.
The models restate the kernels' orders by hand; a change of a kernel's
protocol must be mirrored here.
"""
import pytest


def _fixpoint(roles, frozen=None, frozen_pos=None):
    sig = set()
    pcs = {r: 0 for r in roles}
    changed = True
    while changed:
        changed = False
        for r, ops in roles.items():
            lim = frozen_pos if r == frozen else len(ops)
            while pcs[r] < lim:
                kind, ev = ops[pcs[r]]
                if kind == "sig":
                    sig.add(ev)
                elif ev not in sig:
                    break
                pcs[r] += 1
                changed = True
    return sig, pcs


def check(roles):
    """Returns (roles that cannot finish, waits that can miss a phase)."""
    _, pcs = _fixpoint(roles)
    dead = [r for r in roles if pcs[r] < len(roles[r])]
    missed = []
    for r, ops in roles.items():
        for pos, (kind, ev) in enumerate(ops):
            if kind == "wait":
                bar, k = ev
                sig, _ = _fixpoint(roles, r, pos)
                if (bar, k + 1) in sig:
                    missed.append((r, pos, ev))
    return dead, missed


def ring(name, i, n):
    """Phase of use i of a ring of n barriers."""
    return ((name, i % n), i // n)


def dprep(nj, n_stages, heads, split_pfull=True):
    """D pre-pass (and the forward's two passes, which run the same protocol):
    nj key blocks, K/V ring of n_stages, `heads` query heads per CTA, S and P
    double-buffered."""
    n_it = nj * heads
    pfull = (lambda t: ring("pfull", t, 2)) if split_pfull else (lambda t: ("pfull", t))
    prod, mma, soft = [], [], []

    def issue(j):
        if j >= n_stages:
            prod.append(("wait", ring("kvempty", j - n_stages, n_stages)))
        prod.append(("sig", ring("kvfull", j, n_stages)))

    if nj:
        issue(0)
    for j in range(nj):
        # three stages: request block j+1 before handing block j over; two: after
        if n_stages >= 3 and j + 1 < nj:
            issue(j + 1)
        prod.append(("wait", ring("kvfull", j, n_stages)))
        prod.append(("sig", ring("kvready", j, n_stages)))
        if n_stages < 3 and j + 1 < nj:
            issue(j + 1)

    def pv(t):
        mma.append(("wait", pfull(t)))
        if t % heads == heads - 1:
            mma.append(("sig", ring("kvempty", t // heads, n_stages)))
        mma.append(("sig", ring("pempty", t, 2)))

    for it in range(n_it):
        if it % heads == 0:
            mma.append(("wait", ring("kvready", it // heads, n_stages)))
        mma.append(("sig", ring("sfull", it, 2)))
        if it > 0:
            pv(it - 1)
    if n_it:
        pv(n_it - 1)
        mma.append(("sig", ("ofull", 0)))
    for it in range(n_it):
        soft.append(("wait", ring("sfull", it, 2)))
        if it >= 2:
            soft.append(("wait", ring("pempty", it - 2, 2)))
        soft.append(("sig", pfull(it)))
    if n_it:
        soft.append(("wait", ("ofull", 0)))
    return {"producer": prod, "mma": mma, "softmax": soft}


def _q_producer(n):
    """Q / dO ring of two stages behind one K/V load (both main kernels)."""
    prod = [("sig", ("kvready", 0))]

    def issue(it):
        if it >= 2:
            prod.append(("wait", ring("qempty", it - 2, 2)))
        prod.append(("sig", ring("qfull", it, 2)))

    if n:
        issue(0)
    for it in range(n):
        prod.append(("wait", ring("qfull", it, 2)))
        prod.append(("sig", ring("qready", it, 2)))
        if it + 1 < n:
            issue(it + 1)
    return prod


def main64(n):
    """Main pass, head dim 64: two query halves with their own S/dP and P/dS buffers."""
    mma = [("wait", ("kvready", 0))]
    if n:
        mma += [("wait", ring("qready", 0, 2)), ("sig", (("sfull", 0), 0)), ("sig", (("sfull", 1), 0))]
    for it in range(n):
        more = it + 1 < n
        mma.append(("wait", (("pfull", 0), it)))
        if more:
            mma += [("wait", ring("qready", it + 1, 2)), ("sig", (("sfull", 0), it + 1))]
        mma.append(("wait", (("pfull", 1), it)))
        if it > 0:
            mma.append(("wait", ("dqempty", it - 1)))
        mma += [("sig", ring("qempty", it, 2)), ("sig", ("dqfull", it)),
                ("sig", (("pempty", 0), it)), ("sig", (("pempty", 1), it))]
        if more:
            mma.append(("sig", (("sfull", 1), it + 1)))
    roles = {"producer": _q_producer(n), "mma": mma}
    for g in (0, 1):
        soft = []
        for it in range(n):
            soft.append(("wait", (("sfull", g), it)))
            if it > 0:
                soft.append(("wait", (("pempty", g), it - 1)))
            soft.append(("sig", (("pfull", g), it)))
        roles[f"softmax{g}"] = soft
    roles["epilogue"] = [op for it in range(n) for op in (("wait", ("dqfull", it)), ("sig", ("dqempty", it)))]
    return roles


def main128(n):
    """Main pass, head dim 128: one S/dP buffer, one P/dS tile."""
    mma = [("wait", ("kvready", 0))]
    for it in range(n):
        mma += [("wait", ring("qready", it, 2)), ("sig", ("sfull", it)), ("wait", ("pfull", it))]
        if it > 0:
            mma.append(("wait", ("dqempty", it - 1)))
        mma += [("sig", ring("qempty", it, 2)), ("sig", ("dqfull", it)), ("sig", ("pempty", it))]
    soft = []
    for it in range(n):
        soft.append(("wait", ("sfull", it)))
        if it > 0:
            soft.append(("wait", ("pempty", it - 1)))
        soft.append(("sig", ("pfull", it)))
    epi = [op for it in range(n) for op in (("wait", ("dqfull", it)), ("sig", ("dqempty", it)))]
    return {"producer": _q_producer(n), "mma": mma, "softmax": soft, "epilogue": epi}


@pytest.mark.parametrize("n_stages,heads", [(3, 1), (2, 1), (2, 4)])
def test_dprep_protocol(n_stages, heads):
    for nj in range(0, 10):
        dead, missed = check(dprep(nj, n_stages, heads))
        assert not dead and not missed, (nj, dead, missed[:3])


@pytest.mark.parametrize("fn", [main64, main128])
def test_main_protocols(fn):
    for n in range(0, 12):
        dead, missed = check(fn(n))
        assert not dead and not missed, (n, dead, missed[:3])


def test_single_p_full_barrier_can_miss_a_phase():
    """The check finds the flaw the D pre-pass once had: one P-full barrier for
    both P buffers lets the softmax finish iterations t and t+1 before the MMA
    thread looks at t."""
    for n_stages, heads in [(3, 1), (2, 4)]:
        dead, missed = check(dprep(4, n_stages, heads, split_pfull=False))
        assert not dead
        assert any(ev[0] == "pfull" for _, _, ev in missed)
