"""Models of the mbarrier protocols of the tcgen05 kernels, checked on the
CPU: the attention kernels (sparse_backward_gemm_gb300/csrc/attn.cu) and the
GEMM in its two forms (lone CTAs, 2-SM pairs;
sparse_backward_gemm_gb300/csrc/gemm_tc.cu).

Each role of a kernel (TMA producer, MMA issuer, softmax warps, epilogue and
reducer warps) is written as its sequence of operations on (barrier, phase) events:
  sig     a single-arrival completion (a TMA transaction, a tcgen05.commit,
          a one-thread arrive)
  arrive  one of several arrivals a phase needs (warps of a group); the
          phase completes when every listed arriver has arrived
  wait    block until the phase has completed
Three properties are checked for every sequence length:
  * no deadlock: run to quiescence, every role finishes;
  * no missed phase: every mbarrier wait is a parity wait, so a wait for
    phase k must never find phase k+1 already complete (the parity would
    read as "not yet" and the wait would run out);
  * no overrun: an arriver must never arrive for phase k+1 of a barrier
    while another arriver's arrival for phase k is still pending (the early
    arrival would be counted toward phase k and complete it too soon).
Both hazards are checked by freezing one role just before the operation in
question while every other role runs as far as it can.  Warps are modelled
one by one where a barrier counts several of them; a named barrier (bar.sync)
is an arrive followed by a wait.  The models restate the kernels' orders by
hand; a change of a kernel's protocol must be mirrored here.
"""
import pytest


def _run(roles, arrivers, frozen=None, frozen_pos=None):
    done, arrived = set(), set()
    pcs = {r: 0 for r in roles}
    changed = True
    while changed:
        changed = False
        for r, ops in roles.items():
            lim = frozen_pos if r == frozen else len(ops)
            while pcs[r] < lim:
                kind, ev = ops[pcs[r]]
                if kind == "sig":
                    done.add(ev)
                elif kind == "arrive":
                    bar, k = ev
                    arrived.add((bar, k, r))
                    if all((bar, k, a) in arrived for a in arrivers[bar]):
                        done.add(ev)
                elif ev not in done:
                    break
                pcs[r] += 1
                changed = True
    return done, arrived, pcs


def check(model):
    """Returns (roles that cannot finish, waits that can miss a phase, arrivals that can overrun)."""
    roles, arrivers = model
    _, _, pcs = _run(roles, arrivers)
    dead = [r for r in roles if pcs[r] < len(roles[r])]
    missed, overrun = [], []
    for r, ops in roles.items():
        for pos, (kind, (bar, k)) in enumerate(ops):
            if kind == "wait" and not (isinstance(bar, tuple) and bar[0] == "nb"):
                done, _, _ = _run(roles, arrivers, r, pos)
                if (bar, k + 1) in done:
                    missed.append((r, pos, (bar, k)))
            if kind == "arrive":
                _, arrived, _ = _run(roles, arrivers, r, pos)
                if any((bar, k + 1, a) in arrived for a in arrivers[bar] if a != r):
                    overrun.append((r, pos, (bar, k)))
    return dead, missed, overrun


def ring(name, i, n):
    """Phase of use i of a ring of n barriers."""
    return ((name, i % n), i // n)


def dprep(nj, n_stages, heads, split_pfull=True, warps=2):
    """D pre-pass (and the forward's two passes, which run the same protocol):
    nj key blocks, K/V ring of n_stages, `heads` query heads per CTA, S and P
    double-buffered; the softmax warps arrive on P-full without a named
    barrier between iterations."""
    n_it = nj * heads
    pfull = (lambda t: ring("pfull", t, 2)) if split_pfull else (lambda t: ("pfull", t))
    prod, mma = [], []

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
    roles = {"producer": prod, "mma": mma}
    soft_names = [f"softmax{w}" for w in range(warps)]
    for name in soft_names:
        soft = []
        for it in range(n_it):
            soft.append(("wait", ring("sfull", it, 2)))
            if it >= 2:
                soft.append(("wait", ring("pempty", it - 2, 2)))
            soft.append(("arrive", pfull(it)))
        if n_it:
            soft.append(("wait", ("ofull", 0)))
        roles[name] = soft
    bars = [("pfull", 0), ("pfull", 1)] if split_pfull else ["pfull"]
    return roles, {b: soft_names for b in bars}


def _q_producer(n, stages=2):
    """Q / dO ring behind one K/V load: block it + stages - 1 is requested once
    block it is handed over (both main passes use two stages)."""
    prod = [("sig", ("kvready", 0))]

    def issue(it):
        if it >= stages:
            prod.append(("wait", ring("qempty", it - stages, stages)))
        prod.append(("sig", ring("qfull", it, stages)))

    for it in range(min(stages - 1, n)):
        issue(it)
    for it in range(n):
        prod.append(("wait", ring("qfull", it, stages)))
        prod.append(("sig", ring("qready", it, stages)))
        if it + stages - 1 < n:
            issue(it + stages - 1)
    return prod


def main64(n, warps=2):
    """Main pass, head dim 64: two query halves, each with its own S/dP buffer
    (where its P lands too) and group of softmax warps (a named barrier per
    block); the dS^T tile and the dQ accumulator are double-buffered by block,
    so a half waits only for the dQ of two blocks back; Q / dO have two stages.
    The epilogue warps drain dQ into two staging boxes and hand them to the
    reducer of the block's parity (one thread each), which hands them back
    once its reduce-add has read them."""
    mma = [("wait", ("kvready", 0))]
    if n:
        mma += [("wait", ring("qready", 0, 2)), ("sig", (("sfull", 0), 0)), ("sig", (("sfull", 1), 0))]
    for it in range(n):
        more = it + 1 < n
        mma.append(("wait", (("pfull", 0), it)))
        if more:
            mma += [("wait", ring("qready", it + 1, 2)), ("sig", (("sfull", 0), it + 1))]
        mma.append(("wait", (("pfull", 1), it)))
        mma.append(("sig", ring("qempty", it, 2)))
        if it >= 2:
            mma.append(("wait", ring("dqempty", it - 2, 2)))
        mma += [("sig", ring("dqfull", it, 2)), ("sig", ring("dsempty", it, 2))]
        if more:
            mma.append(("sig", (("sfull", 1), it + 1)))
    roles = {"producer": _q_producer(n, 2), "mma": mma}
    arrivers = {}
    for g in (0, 1):
        names = [f"softmax{g}.{w}" for w in range(warps)]
        for name in names:
            ops = []
            for it in range(n):
                ops += [("arrive", (("nb", g), it)), ("wait", (("nb", g), it)), ("wait", (("sfull", g), it))]
                if it >= 2:
                    ops.append(("wait", ring("dsempty", it - 2, 2)))
                ops.append(("arrive", (("pfull", g), it)))
            roles[name] = ops
        arrivers[("pfull", g)] = names
        arrivers[("nb", g)] = names
    names = [f"epilogue{w}" for w in range(2)]
    for name in names:
        ops = []
        for it in range(n):
            ops.append(("wait", ring("dqfull", it, 2)))
            if it > 0:
                ops.append(("wait", ring("boxfree", it - 1, 2)))
            ops += [("arrive", ring("dqempty", it, 2)), ("arrive", (("nb", "epi"), it)), ("wait", (("nb", "epi"), it))]
            if name == "epilogue0":
                ops.append(("sig", ring("staged", it, 2)))
        if n:   # dK, dV through the dS^T buffers
            ops += [("arrive", (("nb", "epi"), n)), ("wait", (("nb", "epi"), n))]
        roles[name] = ops
    for a in (0, 1):
        arrivers[("dqempty", a)] = names
    arrivers[("nb", "epi")] = names
    for r in (0, 1):
        roles[f"reducer{r}"] = [op for it in range(r, n, 2)
                                for op in (("wait", ring("staged", it, 2)), ("sig", ring("boxfree", it, 2)))]
    return roles, arrivers


def main128(n, warps=2):
    """Main pass, head dim 128: one S/dP buffer (where P and dS land too), the
    softmax warps meet at a named barrier per block; the next block's S, dP
    are issued before this block's dQ^T, and the dS^T tile is double-buffered
    by block for dQ^T.  dQ^T goes through one staging area to the reducer of
    the block's parity, as in the head-dim-64 pass."""
    mma = [("wait", ("kvready", 0))]
    if n:
        mma += [("wait", ring("qready", 0, 2)), ("sig", ("sfull", 0))]
    for it in range(n):
        mma += [("wait", ("pfull", it)), ("sig", ring("qempty", it, 2))]
        if it + 1 < n:
            mma += [("wait", ring("qready", it + 1, 2)), ("sig", ("sfull", it + 1))]
        if it > 0:
            mma.append(("wait", ("dqempty", it - 1)))
        mma += [("sig", ("dqfull", it)), ("sig", ring("dsempty", it, 2))]
    roles = {"producer": _q_producer(n), "mma": mma}
    names = [f"softmax{w}" for w in range(warps)]
    for name in names:
        ops = []
        for it in range(n):
            ops += [("arrive", (("nb", "soft"), it)), ("wait", (("nb", "soft"), it)), ("wait", ("sfull", it))]
            if it >= 2:
                ops.append(("wait", ring("dsempty", it - 2, 2)))
            ops.append(("arrive", ("pfull", it)))
        roles[name] = ops
    arrivers = {"pfull": names, ("nb", "soft"): names}
    # epilogue: drain dQ^T, hand the accumulator back, stage it once the
    # previous block's adds have read the boxes, hand it to the reducer of
    # the block's parity (one thread each)
    enames = [f"epilogue{w}" for w in range(2)]
    for name in enames:
        ops = []
        for it in range(n):
            ops += [("wait", ("dqfull", it)), ("arrive", ("dqempty", it))]
            if it > 0:
                ops.append(("wait", ring("boxfree", it - 1, 2)))
            ops += [("arrive", (("nb", "epi"), it)), ("wait", (("nb", "epi"), it))]
            if name == "epilogue0":
                ops.append(("sig", ring("staged", it, 2)))
        if n:   # dK, dV through the same boxes, once the last adds have read them
            ops.append(("wait", ring("boxfree", n - 1, 2)))
        roles[name] = ops
    arrivers["dqempty"] = enames
    arrivers[("nb", "epi")] = enames
    for r in (0, 1):
        roles[f"reducer{r}"] = [op for it in range(r, n, 2)
                                for op in (("wait", ring("staged", it, 2)), ("sig", ring("boxfree", it, 2)))]
    return roles, arrivers


@pytest.mark.parametrize("n_stages,heads", [(3, 1), (2, 1), (2, 4)])
def test_dprep_protocol(n_stages, heads):
    for nj in range(0, 9):
        dead, missed, overrun = check(dprep(nj, n_stages, heads))
        assert not dead and not missed and not overrun, (nj, dead, missed[:3], overrun[:3])


@pytest.mark.parametrize("fn", [main64, main128])
def test_main_protocols(fn):
    for n in range(0, 10):
        dead, missed, overrun = check(fn(n))
        assert not dead and not missed and not overrun, (n, dead, missed[:3], overrun[:3])


def test_single_p_full_barrier_is_unsafe():
    """The check finds the flaw the D pre-pass once had.  With one P-full
    barrier for both P buffers, the softmax can finish iterations t and t+1
    before the MMA thread looks at t (a missed phase).  And one warp can
    arrive for t+1 before another has arrived for t (an overrun)."""
    for n_stages, heads in [(3, 1), (2, 4)]:
        dead, missed, overrun = check(dprep(4, n_stages, heads, split_pfull=False))
        assert not dead
        assert any(ev[0] == "pfull" for _, _, ev in missed)
        assert any(ev[0] == "pfull" for _, _, ev in overrun)


# ---------------------------------------------------------------------------
# tcgen05 GEMM (sparse_backward_gemm_gb300/csrc/gemm_tc.cu): an S-stage ring
# of shared-memory stages, a double-buffered TMEM accumulator, epilogue warps
# that release it.  `tiles` whole tiles of `kb` k-blocks each.
def gemm(mode, tiles, kb, S, warps=2, segs=None):
    """segs: k-blocks of each segment (a whole tile, or a stream-K piece of
    one); default `tiles` segments of `kb`."""
    segs = [kb] * tiles if segs is None else list(segs)
    tiles = len(segs)
    starts = [sum(segs[:i]) for i in range(tiles)]
    G = sum(segs)
    roles, arrivers = {}, {}
    ctas = ["A"] if mode == 0 else ["A", "B"]
    for c in ctas:
        ops = []
        for g in range(G):
            if g >= S:
                ops.append(("wait", ring(("empty", c), g - S, S)))
            if mode == 0:
                ops.append(("sig", ring(("full", c), g, S)))
            else:
                # every copy of both CTAs is counted on the even CTA's full barrier
                ops.append(("arrive", ring(("full", "A"), g, S)))
        if mode != 0:
            # a pair member leaves only after both MMAs released every stage it loaded
            ops += [("wait", ring(("empty", c), g, S)) for g in range(max(0, G - S), G)]
        roles[f"producer{c}"] = ops
    if mode == 2:
        for s in range(S):
            arrivers[(("full", "A"), s)] = [f"producer{c}" for c in ctas]
    issuers = ctas if mode != 2 else ["A"]     # 2-SM: the even CTA issues for both
    for c in issuers:
        ops = []
        for t in range(tiles):
            if t >= 2:
                ops.append(("wait", ring(("tempty", c), t - 2, 2)))
            for k in range(segs[t]):
                g = starts[t] + k
                ops.append(("wait", ring(("full", c), g, S)))
                if mode == 0:
                    ops.append(("sig", ring(("empty", c), g, S)))
                else:
                    ops += [("sig", ring(("empty", x), g, S)) for x in ctas]
            ops += [("sig", ring(("tfull", x), t, 2)) for x in (ctas if mode == 2 else [c])]
        roles[f"mma{c}"] = ops
    epi_names = {c: [f"epilogue{c}.{w}" for w in range(warps)] for c in ctas}
    for c in ctas:
        owner = "A" if mode == 2 else c          # 2-SM: both epilogues release on the even CTA
        for name in epi_names[c]:
            ops = []
            for t in range(tiles):
                ops += [("wait", ring(("tfull", c), t, 2)), ("arrive", ring(("tempty", owner), t, 2))]
            roles[name] = ops
    for c in issuers:
        names = [n for x in ctas for n in epi_names[x]] if mode == 2 else epi_names[c]
        for a in range(2):
            arrivers[(("tempty", c), a)] = names
    return roles, arrivers


@pytest.mark.parametrize("mode", [0, 2])
def test_gemm_protocols(mode):
    for tiles in range(0, 5):
        for kb in (1, 2, 5):
            for S in (2, 3, 7):
                dead, missed, overrun = check(gemm(mode, tiles, kb, S))
                assert not dead and not missed and not overrun, (mode, tiles, kb, S, dead, missed[:2], overrun[:2])


@pytest.mark.parametrize("mode", [0, 2])
def test_gemm_protocols_with_stream_k_segments(mode):
    """Stream-K gives a CTA (or pair) segments of unequal length: the same
    protocol, with a varying number of k-blocks between accumulator hand-offs."""
    import random
    rnd = random.Random(5)
    for _ in range(40):
        segs = [rnd.randint(1, 6) for _ in range(rnd.randint(1, 5))]
        for S in (2, 3, 7):
            dead, missed, overrun = check(gemm(mode, 0, 0, S, segs=segs))
            assert not dead and not missed and not overrun, (mode, segs, S, dead, missed[:2], overrun[:2])


def test_checker_catches_planted_gemm_flaws():
    """Dropping a wait from a correct model must be caught."""
    # the MMA issuer no longer waits for the epilogues to release the accumulator
    roles, arrivers = gemm(2, 4, 2, 3)
    roles["mmaA"] = [op for op in roles["mmaA"] if not (op[0] == "wait" and op[1][0][0][0] == "tempty")]
    dead, missed, overrun = check((roles, arrivers))
    assert missed and overrun
    # the producers no longer wait for a stage to be consumed
    roles, arrivers = gemm(2, 3, 2, 2)
    for c in "AB":
        roles[f"producer{c}"] = [op for op in roles[f"producer{c}"] if op[0] != "wait"]
    dead, missed, overrun = check((roles, arrivers))
    assert missed and overrun
