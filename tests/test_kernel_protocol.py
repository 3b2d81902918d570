"""A model of the attention kernel's mbarrier protocol, run on the CPU.

Each warp role of the kernel (query/key producer, value producer, S issuer,
P V issuer, softmax, epilogue) is a generator of the same waits and arrivals,
with the same parities, as its device code; the tensor pipe completes queued
MMA commits in order after random delays.  Over random unit sequences and
random interleavings the model checks that no role deadlocks, that every
parity wait passes only once the awaited phase has completed, and that no
wait ever faces a barrier two phases ahead (where a parity check would read
the wrong phase)."""
import random

import pytest


class _Bar:
    def __init__(self, name):
        self.name, self.c = name, 0  # c: completed phases (count 1: one arrival each)

    def arrive(self):
        self.c += 1


def _run(units, kst, vst, seed, rare, handover_wait=True, precise=False):
    rng = random.Random(seed)
    B = {}
    for i in range(2):
        for nm in ("QFull", "QEmpty", "SFull", "SFree", "PReady", "PvDone", "PRead"):
            B[f"{nm}{i}"] = _Bar(f"{nm}{i}")
    for i in range(kst):
        B[f"KFull{i}"], B[f"KEmpty{i}"] = _Bar("KFull"), _Bar("KEmpty")
    for i in range(vst):
        B[f"VFull{i}"], B[f"VEmpty{i}"] = _Bar("VFull"), _Bar("VEmpty")
    for nm in ("OFree", "LmFull", "LmFree"):
        B[nm] = _Bar(nm)
    pipe = []
    posted = {0: None, 1: None}  # precise path: the tile whose rescale factor waits, per parity

    def W(n, par, k):  # wait for phase k of n (parity par)
        return ("wait", n, par, k)

    def A(n):
        return ("arrive", n)

    def producer_qk():
        g = 0
        for u, n in enumerate(units):
            qb = u & 1
            yield W(f"QEmpty{qb}", ((u >> 1) & 1) ^ 1, (u >> 1) - 1)
            yield A(f"QFull{qb}")
            for _ in range(n):
                st = g % kst
                yield W(f"KEmpty{st}", ((g // kst) & 1) ^ 1, g // kst - 1)
                yield A(f"KFull{st}")
                g += 1

    def producer_v():
        g = 0
        for n in units:
            for _ in range(n):
                st = g % vst
                yield W(f"VEmpty{st}", ((g // vst) & 1) ^ 1, g // vst - 1)
                yield A(f"VFull{st}")
                g += 1

    def mma_s():
        t = 0
        for u, n in enumerate(units):
            qb = u & 1
            yield W(f"QFull{qb}", (u >> 1) & 1, u >> 1)
            for j in range(n):
                k, b = t % kst, t & 1
                yield W(f"KFull{k}", (t // kst) & 1, t // kst)
                if t >= 2:
                    yield W(f"SFree{b}", ((t >> 1) - 1) & 1, (t >> 1) - 1)
                yield ("mma", [f"SFull{b}", f"KEmpty{k}"] + ([f"QEmpty{qb}"] if j + 1 == n else []))
                t += 1

    def mma_pv():
        t = 0
        for u, n in enumerate(units):
            for j in range(n):
                v, b = t % vst, t & 1
                yield W(f"VFull{v}", (t // vst) & 1, t // vst)
                yield W(f"PReady{b}", (t >> 1) & 1, t >> 1)
                if j == 0:
                    yield W("OFree", (u & 1) ^ 1, u - 1)
                yield ("mma", [f"PvDone{b}", f"VEmpty{v}"])
                t += 1

    def softmax():
        t = 0
        for u, n in enumerate(units):
            for j in range(n):
                b = t & 1
                yield W(f"SFull{b}", (t >> 1) & 1, t >> 1)
                yield A(f"SFree{b}")
                if j > 0 and rng.random() < rare:  # rescale O after P(t-1) V(t-1)
                    yield W(f"PvDone{(t - 1) & 1}", ((t - 1) >> 1) & 1, (t - 1) >> 1)
                    if precise:  # post the factor once the epilogue has summed P(t-1)
                        yield W(f"PRead{(t - 1) & 1}", ((t - 1) >> 1) & 1, (t - 1) >> 1)
                        assert posted[b] is None, "a posted factor was overwritten"
                        posted[b] = t
                if t >= 2:  # P buffer b free: P(t-2) V(t-2) done (and, precise, summed)
                    yield W(f"PvDone{b}", ((t >> 1) - 1) & 1, (t >> 1) - 1)
                    if precise:
                        yield W(f"PRead{b}", ((t >> 1) - 1) & 1, (t >> 1) - 1)
                yield A(f"PReady{b}")
                t += 1
            if u > 0:
                yield W("LmFree", (u - 1) & 1, u - 1)
            yield A("LmFull")

    def epilogue():
        t = 0
        for u, n in enumerate(units):
            if precise:  # sum every tile's P as it is handed to the P V product
                for j in range(n):
                    b = (t + j) & 1
                    yield W(f"PReady{b}", ((t + j) >> 1) & 1, (t + j) >> 1)
                    if posted[b] is not None:
                        assert posted[b] == t + j, "the epilogue took another tile's factor"
                        posted[b] = None
                    yield A(f"PRead{b}")
            t += n
            tl = t - 1
            if handover_wait:
                yield W("LmFull", u & 1, u)
            yield A("LmFree")
            yield W(f"PvDone{tl & 1}", (tl >> 1) & 1, tl >> 1)
            yield A("OFree")

    roles = {"qk": producer_qk(), "v": producer_v(), "s": mma_s(), "pv": mma_pv(),
             "softmax": softmax(), "epilogue": epilogue()}
    cur = dict.fromkeys(roles)
    done = set()
    while len(done) < len(roles):
        progressed = False
        if pipe and rng.random() < 0.5:
            for nm in pipe.pop(0):
                B[nm].arrive()
            progressed = True
        order = list(roles)
        rng.shuffle(order)
        for k in order:
            if k in done:
                continue
            if cur[k] is None:
                try:
                    cur[k] = next(roles[k])
                except StopIteration:
                    done.add(k)
                    progressed = True
                    continue
            op = cur[k]
            if op[0] == "arrive":
                B[op[1]].arrive()
                cur[k], progressed = None, True
            elif op[0] == "mma":
                pipe.append(op[1])
                cur[k], progressed = None, True
            else:
                _, nm, par, kk = op
                c = B[nm].c
                if (c & 1) != par:  # what try_wait.parity reports as complete
                    assert c >= kk + 1, f"{k}: wait on {nm} phase {kk} passed early ({c} completed)"
                    cur[k], progressed = None, True
                else:
                    assert c <= kk, f"{k}: wait on {nm} phase {kk} faces phase {c} (aliased)"
        assert progressed or pipe, f"deadlock: { {k: cur[k] for k in roles if k not in done} }"


@pytest.mark.parametrize("precise", [False, True], ids=["default", "precise"])
@pytest.mark.parametrize("kst,vst", [(3, 2), (4, 4), (4, 3)])  # bf16 d=128, d=64, FP8
def test_kernel_barrier_protocol(kst, vst, precise):
    for seed in range(150):
        rng = random.Random(1000 * kst + 10 * vst + seed)
        units = [rng.choice([1, 1, 2, 3, 4, 5, 9, 17]) for _ in range(rng.randint(1, 16))]
        _run(units, kst, vst, seed, rare=rng.choice([0.0, 0.1, 1.0]), precise=precise)


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
