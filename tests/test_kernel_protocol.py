"""A model of the attention kernel's mbarrier protocol, run on the CPU.

Each warp role of the kernel (query/key producer, value producer, S issuer,
P V issuer, softmax, epilogue) is a generator of the same waits and arrivals,
with the same parities, as its device code; the tensor pipe completes queued
MMA commits in order after random delays.  With the fp16 P V product the
epilogue also converts every landed value tile, polling (non-blocking tests)
for whichever of its jobs is ready: the model lets it take any ready one.
Over random unit sequences and random interleavings the model checks that no
role deadlocks, that every parity wait or test passes only once the awaited
phase has completed, and that no wait ever faces a barrier two phases ahead
(where a parity check would read the wrong phase)."""
import random

import pytest


class _Bar:
    def __init__(self, name):
        self.name, self.c = name, 0  # c: completed phases (count 1: one arrival each)

    def arrive(self):
        self.c += 1


def _run(units, kst, vst, seed, rare, handover_wait=True, convert=False):
    rng = random.Random(seed)
    B = {}
    for i in range(2):
        for nm in ("QFull", "QEmpty", "SFull", "SFree", "PReady", "PvDone"):
            B[f"{nm}{i}"] = _Bar(f"{nm}{i}")
    for i in range(kst):
        B[f"KFull{i}"], B[f"KEmpty{i}"] = _Bar("KFull"), _Bar("KEmpty")
    for i in range(vst):
        B[f"VFull{i}"], B[f"VEmpty{i}"] = _Bar("VFull"), _Bar("VEmpty")
        B[f"VConv{i}"] = _Bar("VConv")
    for nm in ("OFree", "LmFull", "LmFree"):
        B[nm] = _Bar(nm)
    pipe = []

    def pv_done(t):  # the P-V-done barrier of tile t (two, alternating) and its phase
        return (f"PvDone{t & 1}", (t >> 1) & 1, t >> 1)

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
                yield W(f"{'VConv' if convert else 'VFull'}{v}", (t // vst) & 1, t // vst)
                yield W(f"PReady{b}", (t >> 1) & 1, t >> 1)
                if j == 0:
                    yield W("OFree", (u & 1) ^ 1, u - 1)
                yield ("mma", [pv_done(t)[0], f"VEmpty{v}"])
                t += 1

    def softmax():
        t = 0
        for u, n in enumerate(units):
            for j in range(n):
                b = t & 1
                yield W(f"SFull{b}", (t >> 1) & 1, t >> 1)
                yield A(f"SFree{b}")
                if j > 0 and rng.random() < rare:  # rescale O after P(t-1) V(t-1)
                    yield W(*pv_done(t - 1))
                if t >= 2:  # P buffer b free: P(t-2) V(t-2) done
                    yield W(*pv_done(t - 2))
                yield A(f"PReady{b}")
                t += 1
            if u > 0:
                yield W("LmFree", (u - 1) & 1, u - 1)
            yield A("LmFull")

    def epilogue():
        t = 0
        for u, n in enumerate(units):
            t += n
            tl = t - 1
            if handover_wait:
                yield W("LmFull", u & 1, u)
            yield A("LmFree")
            yield W(*pv_done(tl))
            yield A("OFree")

    def epilogue_convert():
        # poll whichever job is ready: convert the next landed value tile, or
        # take the pending unit's (m, l), or write it once its last product is done
        total = sum(units)
        tv, go, u, ostage = 0, 0, 0, 0
        while u < len(units) or tv < total:
            opts = []
            if tv < total:
                opts.append((f"VFull{tv % vst}", (tv // vst) & 1, tv // vst, "conv"))
            if u < len(units):
                tl = go + units[u] - 1
                if ostage == 0:
                    opts.append(("LmFull", u & 1, u, "lm"))
                else:
                    opts.append((*pv_done(tl), "out"))
            tag = yield ("poll", opts)
            if tag == "conv":
                yield A(f"VConv{tv % vst}")
                tv += 1
            elif tag == "lm":
                yield A("LmFree")
                ostage = 1
            else:
                yield A("OFree")
                go += units[u]
                u += 1
                ostage = 0

    roles = {"qk": producer_qk(), "v": producer_v(), "s": mma_s(), "pv": mma_pv(),
             "softmax": softmax(), "epilogue": epilogue_convert() if convert else epilogue()}
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
            elif op[0] == "poll":
                ready = []
                for nm, par, kk, tag in op[1]:
                    c = B[nm].c
                    if (c & 1) != par:
                        assert c >= kk + 1, f"{k}: test of {nm} phase {kk} passed early ({c} completed)"
                        ready.append(tag)
                    else:
                        assert c <= kk, f"{k}: test of {nm} phase {kk} faces phase {c} (aliased)"
                if ready:
                    try:
                        cur[k] = roles[k].send(rng.choice(ready))
                    except StopIteration:
                        done.add(k)
                        cur[k] = None
                    progressed = True
            else:
                _, nm, par, kk = op
                c = B[nm].c
                if (c & 1) != par:  # what try_wait.parity reports as complete
                    assert c >= kk + 1, f"{k}: wait on {nm} phase {kk} passed early ({c} completed)"
                    cur[k], progressed = None, True
                else:
                    assert c <= kk, f"{k}: wait on {nm} phase {kk} faces phase {c} (aliased)"
        assert progressed or pipe, f"deadlock: { {k: cur[k] for k in roles if k not in done} }"


@pytest.mark.parametrize("mode", ["bf16_pv", "f16_pv"])
@pytest.mark.parametrize("kst,vst", [(3, 2), (4, 4), (4, 3)])  # bf16 d=128, d=64, FP8
def test_kernel_barrier_protocol(kst, vst, mode):
    for seed in range(150):
        rng = random.Random(1000 * kst + 10 * vst + seed)
        units = [rng.choice([1, 1, 2, 3, 4, 5, 9, 17]) for _ in range(rng.randint(1, 16))]
        _run(units, kst, vst, seed, rare=rng.choice([0.0, 0.1, 1.0]), convert=mode == "f16_pv")


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
