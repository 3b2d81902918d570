"""A model of the attention kernel's mbarrier protocol, run on the CPU.

Each warp role of the kernel (query/key producer, value producer, S issuer,
P V issuer, softmax, epilogue) is a generator of the same waits and arrivals,
with the same parities, as its device code.  TMA copies complete their
barrier after random delays, in any order; the tensor pipe completes queued
MMA commits in order after random delays.  Over random unit sequences and
random interleavings the model checks that no role deadlocks, that every
parity wait passes only once the awaited phase has completed, and that no
wait ever faces a barrier two phases ahead (where a parity check would read
the wrong phase).

The abort path is modelled too: at a random moment a wait runs out of time
and raises the CTA's abort flag.  From then on a wait whose phase has not
completed gives up (as the kernel's bounded waits do), each role leaves its
loop, the producers drain the copies they issued and the MMA issuers commit
and drain their products (drain waits ignore the flag).  When every role has
left, no copy and no MMA may still be in flight: the kernel frees the tensor
memory and the CTA exits at that point."""
import random

import pytest


class _Bar:
    def __init__(self, name, count=1):
        self.name, self.c = name, 0  # c: completed phases
        self.count, self.pending = count, 0

    def arrive(self):
        self.pending += 1
        if self.pending == self.count:
            self.pending = 0
            self.c += 1


def _run(units, kst, vst, seed, rare, handover_wait=True, abort_at=None, pair=False):
    """abort_at: None, or the probability per scheduler round that the abort
    flag is raised (a wait timing out).  pair: the SM-pair kernel, whose
    rank-0 CTA loads and issues for both CTAs: its commits of S and P V reach
    both CTAs' barriers (@0, @1), each CTA's softmax and epilogue wait on
    their own CTA's barriers, and the S-free, P-ready and O-free barriers (on
    rank 0) take one arrival from each CTA's warpgroup."""
    rng = random.Random(seed)
    ranks = (0, 1) if pair else (0,)
    groups = len(ranks)
    B = {}

    def loc(nm, r):  # a barrier each CTA has its own copy of
        return f"{nm}@{r}" if pair else nm

    for i in range(2):
        for nm in ("QFull", "QEmpty", "MmaDone"):
            B[f"{nm}{i}"] = _Bar(f"{nm}{i}")
        for nm in ("SFree", "PReady"):
            B[f"{nm}{i}"] = _Bar(f"{nm}{i}", groups)
        for nm in ("SFull", "PvDone"):
            for r in ranks:
                B[loc(f"{nm}{i}", r)] = _Bar(loc(f"{nm}{i}", r))
    for i in range(kst):
        B[f"KFull{i}"], B[f"KEmpty{i}"] = _Bar("KFull"), _Bar("KEmpty")
    for i in range(vst):
        B[f"VFull{i}"], B[f"VEmpty{i}"] = _Bar("VFull"), _Bar("VEmpty")
    B["OFree"] = _Bar("OFree", groups)
    for r in ranks:
        for nm in ("LmFull", "LmFree"):
            B[loc(nm, r)] = _Bar(loc(nm, r))
    pipe = []      # MMA commits, completed in order
    copies = []    # TMA copies in flight, completed in any order
    state = {"abort": False}

    def pv_done(t, r=0):  # the P-V-done barrier of tile t (two, alternating) and its phase
        return (loc(f"PvDone{t & 1}", r), (t >> 1) & 1, t >> 1)

    def everywhere(nm):  # a commit multicast to both CTAs' copies
        return [loc(nm, r) for r in ranks]

    def W(n, par, k):  # bounded wait for phase k of n (parity par); gives up on abort
        return ("wait", n, par, k)

    def D(n, par, k):  # drain wait: ignores the abort flag
        return ("drain", n, par, k)

    def A(n):
        return ("arrive", n)

    def producer_qk():
        g = k_armed = q_armed = 0
        ok = True
        for u, n in enumerate(units):
            qb = u & 1
            ok = yield W(f"QEmpty{qb}", ((u >> 1) & 1) ^ 1, (u >> 1) - 1)
            if not ok:
                break
            yield ("tma", f"QFull{qb}")
            q_armed += 1
            for _ in range(n):
                st = g % kst
                ok = yield W(f"KEmpty{st}", ((g // kst) & 1) ^ 1, g // kst - 1)
                if not ok:
                    break
                yield ("tma", f"KFull{st}")
                k_armed += 1
                g += 1
            if not ok:
                break
        # let every copy issued land (the latest arming of each stage); after a
        # normal run the consumers have already waited for them all
        for k in range(1, min(kst, k_armed) + 1):
            i = k_armed - k
            yield D(f"KFull{i % kst}", (i // kst) & 1, i // kst)
        for k in range(1, min(2, q_armed) + 1):
            i = q_armed - k
            yield D(f"QFull{i & 1}", (i >> 1) & 1, i >> 1)

    def producer_v():
        g = v_armed = 0
        ok = True
        for n in units:
            for _ in range(n):
                st = g % vst
                ok = yield W(f"VEmpty{st}", ((g // vst) & 1) ^ 1, g // vst - 1)
                if not ok:
                    break
                yield ("tma", f"VFull{st}")
                v_armed += 1
                g += 1
            if not ok:
                break
        for k in range(1, min(vst, v_armed) + 1):
            i = v_armed - k
            yield D(f"VFull{i % vst}", (i // vst) & 1, i // vst)

    def mma_s():
        t = 0
        ok = True
        for u, n in enumerate(units):
            qb = u & 1
            ok = yield W(f"QFull{qb}", (u >> 1) & 1, u >> 1)
            if not ok:
                break
            for j in range(n):
                k, b = t % kst, t & 1
                ok = yield W(f"KFull{k}", (t // kst) & 1, t // kst)
                if ok and t >= 2:
                    ok = yield W(f"SFree{b}", ((t >> 1) - 1) & 1, (t >> 1) - 1)
                if not ok:
                    break
                yield ("mma", everywhere(f"SFull{b}") + [f"KEmpty{k}"] +
                       ([f"QEmpty{qb}"] if j + 1 == n else []))
                t += 1
            if not ok:
                break
        yield ("mma", ["MmaDone0"])  # every MMA of this thread done before TMEM is freed
        yield D("MmaDone0", 0, 0)

    def mma_pv():
        t = 0
        ok = True
        for u, n in enumerate(units):
            for j in range(n):
                v, b = t % vst, t & 1
                ok = yield W(f"VFull{v}", (t // vst) & 1, t // vst)
                if ok:
                    ok = yield W(f"PReady{b}", (t >> 1) & 1, t >> 1)
                if ok and j == 0:
                    ok = yield W("OFree", (u & 1) ^ 1, u - 1)
                if not ok:
                    break
                yield ("mma", everywhere(f"PvDone{t & 1}") + [f"VEmpty{v}"])
                t += 1
            if not ok:
                break
        yield ("mma", ["MmaDone1"])
        yield D("MmaDone1", 0, 0)

    def softmax(r):
        t = 0
        for u, n in enumerate(units):
            for j in range(n):
                b = t & 1
                if not (yield W(loc(f"SFull{b}", r), (t >> 1) & 1, t >> 1)):
                    return
                yield A(f"SFree{b}")
                if j > 0 and rng.random() < rare:  # rescale O after P(t-1) V(t-1)
                    if not (yield W(*pv_done(t - 1, r))):
                        return
                if t >= 2:  # P buffer b free: P(t-2) V(t-2) done
                    if not (yield W(*pv_done(t - 2, r))):
                        return
                yield A(f"PReady{b}")
                t += 1
            if u > 0:
                if not (yield W(loc("LmFree", r), (u - 1) & 1, u - 1)):
                    return
            yield A(loc("LmFull", r))

    def epilogue(r):
        t = 0
        for u, n in enumerate(units):
            t += n
            tl = t - 1
            if handover_wait:
                if not (yield W(loc("LmFull", r), u & 1, u)):
                    return
            yield A(loc("LmFree", r))
            if not (yield W(*pv_done(tl, r))):
                return
            yield A("OFree")

    roles = {"qk": producer_qk(), "v": producer_v(), "s": mma_s(), "pv": mma_pv()}
    for r in ranks:
        roles[f"softmax{r}"] = softmax(r)
        roles[f"epilogue{r}"] = epilogue(r)
    cur = {k: None for k in roles}
    done = set()

    def advance(k, value):
        try:
            cur[k] = roles[k].send(value) if value is not None else next(roles[k])
        except StopIteration:
            cur[k] = None
            done.add(k)

    for k in roles:
        advance(k, None)
    rounds = 0
    while len(done) < len(roles):
        rounds += 1
        assert rounds < 200000, "model did not finish"
        progressed = False
        if abort_at is not None and not state["abort"] and rng.random() < abort_at:
            state["abort"] = True
            progressed = True
        if pipe and rng.random() < 0.5:
            for nm in pipe.pop(0):
                B[nm].arrive()
            progressed = True
        if copies and rng.random() < 0.5:
            B[copies.pop(rng.randrange(len(copies)))].arrive()
            progressed = True
        order = [k for k in roles if k not in done]
        rng.shuffle(order)
        for k in order:
            op = cur[k]
            if op[0] == "arrive":
                B[op[1]].arrive()
                advance(k, True)
                progressed = True
            elif op[0] == "mma":
                pipe.append(op[1])
                advance(k, True)
                progressed = True
            elif op[0] == "tma":
                copies.append(op[1])
                advance(k, True)
                progressed = True
            else:
                kind, nm, par, kk = op
                c = B[nm].c
                if (c & 1) != par:  # what try_wait.parity reports as complete
                    assert c >= kk + 1, f"{k}: wait on {nm} phase {kk} passed early ({c} completed)"
                    advance(k, True)
                    progressed = True
                else:
                    assert c <= kk, f"{k}: wait on {nm} phase {kk} faces phase {c} (aliased)"
                    if kind == "wait" and state["abort"]:
                        advance(k, False)  # the bounded wait gives up
                        progressed = True
        assert progressed or pipe or copies, \
            f"deadlock: { {k: cur[k] for k in roles if k not in done} }"
    # every role has left: the CTA frees TMEM and exits now
    assert not pipe, f"MMAs still in flight at exit: {pipe}"
    assert not copies, f"copies still in flight at exit: {copies}"
    return state["abort"]


@pytest.mark.parametrize("kst,vst", [(3, 2), (4, 4), (4, 3)])  # bf16 d=128, d=64, FP8
def test_kernel_barrier_protocol(kst, vst):
    for seed in range(150):
        rng = random.Random(1000 * kst + 10 * vst + seed)
        units = [rng.choice([1, 1, 2, 3, 4, 5, 9, 17]) for _ in range(rng.randint(1, 16))]
        _run(units, kst, vst, seed, rare=rng.choice([0.0, 0.1, 1.0]))


@pytest.mark.parametrize("kst,vst", [(3, 2), (4, 4), (4, 3)])
def test_abort_path_drains_every_copy_and_mma(kst, vst):
    """Timeouts raised at random moments: every role leaves, and nothing is
    in flight when TMEM is freed."""
    aborted = 0
    for seed in range(300):
        rng = random.Random(7 + 1000 * kst + 10 * vst + seed)
        units = [rng.choice([1, 2, 3, 5, 9, 17]) for _ in range(rng.randint(1, 12))]
        aborted += _run(units, kst, vst, seed, rare=rng.choice([0.0, 0.1, 1.0]),
                        abort_at=rng.choice([0.001, 0.01, 0.1, 0.5]))
    assert aborted >= 150


def test_model_catches_a_missing_drain():
    """Plant a mistake in the model (the producers skip their drain): the
    check that nothing is in flight at exit must catch it."""
    caught = 0
    for seed in range(60):
        rng = random.Random(seed)
        units = [rng.choice([2, 3, 5, 9]) for _ in range(rng.randint(2, 8))]
        try:
            _run_no_drain(units, 3, 2, seed, 0.1, abort_at=0.2)
        except AssertionError as e:
            assert "in flight" in str(e)
            caught += 1
    assert caught >= 10


def _run_no_drain(*args, **kw):
    """_run with the producers' drain waits removed (a planted mistake)."""
    import inspect
    import textwrap
    text = textwrap.dedent(inspect.getsource(_run))
    text = text.replace("yield D(f\"KFull", "pass  # yield D(f\"KFull").replace(
        "yield D(f\"QFull", "pass  # yield D(f\"QFull").replace(
        "yield D(f\"VFull", "pass  # yield D(f\"VFull").replace("def _run(", "def _planted(")
    ns = dict(globals())
    exec(compile(text, "<planted>", "exec"), ns)
    return ns["_planted"](*args, **kw)


def test_model_catches_a_skipped_phase():
    """Without the hand-over wait the epilogue would wait on P-V-done only at
    unit ends, skipping phases; the model must flag the early pass."""
    caught = 0
    for seed in range(40):
        rng = random.Random(seed)
        units = [rng.choice([1, 2, 3, 5, 9]) for _ in range(rng.randint(2, 10))]
        try:
            _run(units, 3, 2, seed, 0.1, handover_wait=False)
        except AssertionError as e:
            assert "passed early" in str(e) or "aliased" in str(e) or "deadlock" in str(e)
            caught += 1
    assert caught >= 30


@pytest.mark.parametrize("kst,vst", [(7, 3), (5, 5)])  # SM-pair rings (16 KB halves)
def test_pair_kernel_barrier_protocol(kst, vst):
    for seed in range(150):
        rng = random.Random(5000 + 10 * kst + vst + seed)
        units = [rng.choice([1, 1, 2, 3, 4, 5, 9, 17]) for _ in range(rng.randint(1, 16))]
        _run(units, kst, vst, seed, rare=rng.choice([0.0, 0.1, 1.0]), pair=True)


@pytest.mark.parametrize("kst,vst", [(7, 3)])
def test_pair_kernel_abort_path_drains_every_copy_and_mma(kst, vst):
    aborted = 0
    for seed in range(300):
        rng = random.Random(9 + 10 * kst + vst + seed)
        units = [rng.choice([1, 2, 3, 5, 9, 17]) for _ in range(rng.randint(1, 12))]
        aborted += _run(units, kst, vst, seed, rare=rng.choice([0.0, 0.1, 1.0]),
                        abort_at=rng.choice([0.001, 0.01, 0.1, 0.5]), pair=True)
    assert aborted >= 150


# ---------------------------------------------------------------------------
# Head-pair clusters: two CTAs, each running every role of the one-CTA kernel
# on its own query head of the same items, share the key and value rings.
# Each CTA's producer arms its own full barrier for the whole tile and copies
# half of it into both CTAs (a multicast copy lands in the two CTAs
# independently); each CTA's MMA issuer commits the stage's empty barrier in
# both CTAs, so a stage is refilled only after both CTAs' products have read
# it.  Barrier events carry the phase they belong to, and the model fails if
# one reaches a barrier whose current phase is another: with two senders per
# ring barrier, that is how a refill racing a slow reader would show.  The
# arrivals a commit makes in the other CTA travel separately and land later.
# Before exiting, each producer waits for its ring's last full and empty
# phases (after an abort those may never complete; the kernel bounds such a
# drain, and the model lets a wait run out only when nothing else can move,
# copies and arrivals landing long before any bound expires).  At the
# cluster barrier nothing may be in flight.

class _TagBar:
    """A barrier whose phase completes after `count` events, each tagged with
    the phase it belongs to."""

    def __init__(self, name, count):
        self.name, self.count, self.c, self.pending = name, count, 0, 0

    def event(self, phase):
        assert phase == self.c, f"{self.name}: event of phase {phase} while phase {self.c} is open"
        self.pending += 1
        if self.pending == self.count:
            self.pending = 0
            self.c += 1


def _run_share(units, kst, vst, seed, rare, abort_at=None, final_empty_wait=True):
    rng = random.Random(seed)
    R = (0, 1)
    B = {}
    for r in R:
        for i in range(2):
            for nm in ("QFull", "QEmpty", "MmaDone", "SFull", "PvDone"):
                B[f"{nm}{i}@{r}"] = _Bar(f"{nm}{i}@{r}")
            for nm in ("SFree", "PReady"):
                B[f"{nm}{i}@{r}"] = _Bar(f"{nm}{i}@{r}")
        for nm in ("OFree", "LmFull", "LmFree"):
            B[f"{nm}@{r}"] = _Bar(f"{nm}@{r}")
        for i in range(kst):
            B[f"KFull{i}@{r}"] = _TagBar(f"KFull{i}@{r}", 3)   # arm + two halves
            B[f"KEmpty{i}@{r}"] = _TagBar(f"KEmpty{i}@{r}", 2)  # both CTAs' commits
        for i in range(vst):
            B[f"VFull{i}@{r}"] = _TagBar(f"VFull{i}@{r}", 3)
            B[f"VEmpty{i}@{r}"] = _TagBar(f"VEmpty{i}@{r}", 2)
    pipes = {r: [] for r in R}  # per CTA: MMA commits, completed in order
    inflight = []   # copies and remote commit arrivals, landing in any order
    abort = {r: False for r in R}

    def hit(target):  # target: name, or (name, phase) for a tagged barrier
        if isinstance(target, tuple):
            B[target[0]].event(target[1])
        else:
            B[target].arrive()

    def W(n, par, k):
        return ("wait", n, par, k)

    def D(n, par, k):
        return ("drain", n, par, k)

    def producer(r, ring, stages, with_q):
        g = armed = q_armed = 0
        ok = True
        for u, n in enumerate(units):
            if with_q:
                qb = u & 1
                ok = yield W(f"QEmpty{qb}@{r}", ((u >> 1) & 1) ^ 1, (u >> 1) - 1)
                if not ok:
                    break
                yield ("copy", [f"QFull{qb}@{r}"])
                q_armed += 1
            for _ in range(n):
                st, ph = g % stages, g // stages
                ok = yield W(f"{ring}Empty{st}@{r}", (ph & 1) ^ 1, ph - 1)
                if not ok:
                    break
                yield ("arrive", (f"{ring}Full{st}@{r}", ph))
                yield ("copy", [(f"{ring}Full{st}@{x}", ph) for x in R])
                armed += 1
                g += 1
            if not ok:
                break
        for k in range(1, min(stages, armed) + 1):
            i = armed - k
            yield D(f"{ring}Full{i % stages}@{r}", (i // stages) & 1, i // stages)
        for k in range(1, min(2, q_armed) + 1):
            i = q_armed - k
            yield D(f"QFull{i & 1}@{r}", (i >> 1) & 1, i >> 1)
        if final_empty_wait:  # the other CTA's last commits have landed here
            for k in range(1, min(stages, armed) + 1):
                i = armed - k
                yield D(f"{ring}Empty{i % stages}@{r}", (i // stages) & 1, i // stages)

    def mma_s(r):
        t = 0
        ok = True
        for u, n in enumerate(units):
            qb = u & 1
            ok = yield W(f"QFull{qb}@{r}", (u >> 1) & 1, u >> 1)
            if not ok:
                break
            for j in range(n):
                k, b, ph = t % kst, t & 1, t // kst
                ok = yield W(f"KFull{k}@{r}", ph & 1, ph)
                if ok and t >= 2:
                    ok = yield W(f"SFree{b}@{r}", ((t >> 1) - 1) & 1, (t >> 1) - 1)
                if not ok:
                    break
                yield ("mma", [f"SFull{b}@{r}"] + [(f"KEmpty{k}@{x}", ph) for x in R] +
                       ([f"QEmpty{qb}@{r}"] if j + 1 == n else []))
                t += 1
            if not ok:
                break
        yield ("mma", [f"MmaDone0@{r}"])
        yield D(f"MmaDone0@{r}", 0, 0)

    def mma_pv(r):
        t = 0
        ok = True
        for u, n in enumerate(units):
            for j in range(n):
                v, b, ph = t % vst, t & 1, t // vst
                ok = yield W(f"VFull{v}@{r}", ph & 1, ph)
                if ok:
                    ok = yield W(f"PReady{b}@{r}", (t >> 1) & 1, t >> 1)
                if ok and j == 0:
                    ok = yield W(f"OFree@{r}", (u & 1) ^ 1, u - 1)
                if not ok:
                    break
                yield ("mma", [f"PvDone{b}@{r}"] + [(f"VEmpty{v}@{x}", ph) for x in R])
                t += 1
            if not ok:
                break
        yield ("mma", [f"MmaDone1@{r}"])
        yield D(f"MmaDone1@{r}", 0, 0)

    def softmax(r):
        t = 0
        for u, n in enumerate(units):
            for j in range(n):
                b = t & 1
                if not (yield W(f"SFull{b}@{r}", (t >> 1) & 1, t >> 1)):
                    return
                yield ("arrive", f"SFree{b}@{r}")
                if j > 0 and rng.random() < rare:
                    tp = t - 1
                    if not (yield W(f"PvDone{tp & 1}@{r}", (tp >> 1) & 1, tp >> 1)):
                        return
                if t >= 2:
                    tp = t - 2
                    if not (yield W(f"PvDone{tp & 1}@{r}", (tp >> 1) & 1, tp >> 1)):
                        return
                yield ("arrive", f"PReady{b}@{r}")
                t += 1
            if u > 0:
                if not (yield W(f"LmFree@{r}", (u - 1) & 1, u - 1)):
                    return
            yield ("arrive", f"LmFull@{r}")

    def epilogue(r):
        t = 0
        for u, n in enumerate(units):
            t += n
            tl = t - 1
            if not (yield W(f"LmFull@{r}", u & 1, u)):
                return
            yield ("arrive", f"LmFree@{r}")
            if not (yield W(f"PvDone{tl & 1}@{r}", (tl >> 1) & 1, tl >> 1)):
                return
            yield ("arrive", f"OFree@{r}")

    roles = {}
    for r in R:
        roles[(r, "qk")] = producer(r, "K", kst, True)
        roles[(r, "v")] = producer(r, "V", vst, False)
        roles[(r, "s")] = mma_s(r)
        roles[(r, "pv")] = mma_pv(r)
        roles[(r, "softmax")] = softmax(r)
        roles[(r, "epilogue")] = epilogue(r)
    cur = {k: None for k in roles}
    done = set()

    def advance(k, value):
        try:
            cur[k] = roles[k].send(value) if value is not None else next(roles[k])
        except StopIteration:
            cur[k] = None
            done.add(k)

    for k in roles:
        advance(k, None)
    rounds = 0
    while len(done) < len(roles):
        rounds += 1
        assert rounds < 400000, "model did not finish"
        progressed = False
        for r in R:
            if abort_at is not None and not abort[r] and rng.random() < abort_at:
                abort[r] = progressed = True
            if pipes[r] and rng.random() < 0.5:
                targets = pipes[r].pop(0)
                for tg in targets:  # this CTA's barriers now, the other CTA's later
                    if isinstance(tg, tuple) and not tg[0].endswith(f"@{r}"):
                        inflight.append(tg)
                    else:
                        hit(tg)
                progressed = True
        if inflight and rng.random() < 0.5:
            hit(inflight.pop(rng.randrange(len(inflight))))
            progressed = True
        order = [k for k in roles if k not in done]
        rng.shuffle(order)
        stuck = []
        for k in order:
            r, op = k[0], cur[k]
            if op[0] == "arrive":
                hit(op[1])
                advance(k, True)
                progressed = True
            elif op[0] == "mma":
                pipes[r].append(op[1])
                advance(k, True)
                progressed = True
            elif op[0] == "copy":
                inflight.extend(op[1])
                advance(k, True)
                progressed = True
            else:
                kind, nm, par, kk = op
                c = B[nm].c
                if (c & 1) != par:
                    assert c >= kk + 1, f"{k}: wait on {nm} phase {kk} passed early ({c} completed)"
                    advance(k, True)
                    progressed = True
                else:
                    assert c <= kk, f"{k}: wait on {nm} phase {kk} faces phase {c} (aliased)"
                    if kind == "wait" and abort[r]:
                        advance(k, False)
                        progressed = True
                    else:
                        stuck.append(k)
        if not progressed and not inflight and not any(pipes.values()):
            # Nothing can move: a bounded wait runs out (a drain wait after
            # its own, longer, limit) and its CTA aborts.
            assert stuck, "deadlock with no waiter"
            assert abort_at is not None, f"deadlock: { {k: cur[k] for k in stuck} }"
            k = stuck[0]
            abort[k[0]] = True
            advance(k, False)
    # both CTAs have left every role; they pass the cluster barrier and exit
    assert not any(pipes.values()), f"MMAs still in flight at exit: {pipes}"
    assert not inflight, f"copies or arrivals still in flight at exit: {inflight}"
    return abort[0] or abort[1]


@pytest.mark.parametrize("kst,vst", [(2, 3), (5, 3), (4, 4), (3, 2)])  # bf16, FP8 q/k, d 64; other
def test_share_cluster_barrier_protocol(kst, vst):
    for seed in range(120):
        rng = random.Random(7000 + 10 * kst + vst + seed)
        units = [rng.choice([1, 1, 2, 3, 4, 5, 9, 17]) for _ in range(rng.randint(1, 16))]
        assert not _run_share(units, kst, vst, seed, rare=rng.choice([0.0, 0.1, 1.0]))


@pytest.mark.parametrize("kst,vst", [(2, 3), (5, 3)])
def test_share_cluster_abort_path(kst, vst):
    """Timeouts at random moments in either CTA: both CTAs leave, and nothing
    is in flight when they pass the cluster barrier."""
    aborted = 0
    for seed in range(250):
        rng = random.Random(11 + 10 * kst + vst + seed)
        units = [rng.choice([1, 2, 3, 5, 9, 17]) for _ in range(rng.randint(1, 12))]
        aborted += _run_share(units, kst, vst, seed, rare=rng.choice([0.0, 0.1, 1.0]),
                              abort_at=rng.choice([0.001, 0.01, 0.1, 0.5]))
    assert aborted >= 120


def test_share_model_catches_a_missing_final_wait():
    """Plant a mistake (the producers skip the wait for the other CTA's last
    commits): some run must end with an arrival still in flight."""
    caught = 0
    for seed in range(80):
        rng = random.Random(300 + seed)
        units = [rng.choice([1, 2, 3, 5]) for _ in range(rng.randint(1, 6))]
        try:
            _run_share(units, 2, 3, seed, 0.1, final_empty_wait=False)
        except AssertionError as e:
            assert "in flight" in str(e)
            caught += 1
    assert caught >= 10
