"""Host model of the synchronisation protocol of the column-block dense compose kernel
(csrc/compose_cols.cu): a CTA takes (unit, block of state columns) tiles, n segments each.

Roles, as in the kernel: the four split warps (each its rows of A of every MMA step, P_j as tf32 hi and lo parts in
TMEM, k-block by k-block as the previous step's products release it; once all four warps
have read a P stage, one of them refills it with the P two MMA steps on); four MMA issuers
(issuer i: k-step i of every k-block, its three products, into its own accumulator D_i; a
k-block goes back once all four issuers' products on it have completed); and the epilogue
warps (D = the sum of the D_i, D + S_j -> the prefix state; X_j, the next step's B operand,
written over X_{j-1}; X from S0 at a tile's start; prefix_j written over S_j in its slot and
stored by one bulk tensor store, after which thread 0 refills the previous step's slot, its
store having read it, with the S four steps on). The copy engine lands loads in issue order
at random times. Each group of warps that arrives and waits together is one agent; the
tensor pipe runs each issuer's products in order, and a commit fires once every product its
issuer issued before it has completed.

Every run checks for deadlock, parity aliasing, and that every buffer (P stages, S slots, A
k-blocks, X, D) is read in the version its reader needs and never overwritten under a reader.
It runs on the CPU only.
"""
import random

import pytest


class Hazard(Exception):
    pass


class _Bar:
    def __init__(self, count=1):
        self.count, self.arr, self.done = count, 0, 0

    def arrive(self):
        self.arr += 1
        if self.arr == self.count:
            self.arr = 0
            self.done += 1


def _run(ns, s0, seed, mistake=None, tiles=1, stages=2, s_slots=4):
    rnd = random.Random(seed)
    # the steps of every tile a CTA takes, in order; a step with a carried state runs products
    steps = [(t, j) for t in range(tiles) for j in range(ns)]
    mma_steps = [(t, j) for (t, j) in steps if j > 0 or s0]
    B = {"xfull": _Bar(), "dfull": _Bar(4)}
    for i in range(stages):
        B[f"pfull{i}"], B[f"pempty{i}"] = _Bar(), _Bar(4)
    for i in range(4):
        B[f"afull{i}"], B[f"aempty{i}"] = _Bar(4), _Bar(4)
    for i in range(s_slots):
        B[f"sfull{i}"] = _Bar()
    m = dict(P={}, Preading={}, A={}, X=None, D={}, S={}, Sreading={})
    queues, inflight, commits = [[] for _ in range(4)], [[] for _ in range(4)], [[] for _ in range(4)]
    started, done, stores, loads = [0] * 4, [0] * 4, [], []

    def wait(name, phase):
        b = B[name]
        if b.done > phase + 1:
            raise Hazard(f"parity alias on {name}")
        while b.done <= phase:
            yield

    def prev(step):
        t, j = step
        return (t, j - 1) if j > 0 else (t, "S0")

    def rw(op):
        reads = {("A", (op["b"], w)): op["step"] for w in range(4)}
        reads["X"] = prev(op["step"])
        return reads, {("D", op["i"]): op["step"]}

    def touches(keys, writing, who):
        for x in (y for q in inflight for y in q):
            r, w = rw(x)
            if any(k in w for k in keys) or (writing and any(k in r for k in keys)):
                raise Hazard(f"{who} touches {keys} under the in-flight MMA of step {x['step']}")

    def load_p(pc):
        if pc < len(mma_steps):
            loads.append(("P", pc % stages, mma_steps[pc]))

    def load_s(sc):
        if sc < len(steps):
            loads.append(("S", sc % s_slots, steps[sc]))

    def tma():
        # the copy engine: the loads issued so far land in order, some time later
        while True:
            if loads and rnd.random() < 0.3:
                kind, slot, step = loads.pop(0)
                if kind == "P":
                    if any(m["Preading"].get((slot, w)) for w in range(4)):
                        raise Hazard("P stage overwritten while the split reads it")
                    m["P"][slot] = step
                    B[f"pfull{slot}"].arrive()
                else:
                    if m["Sreading"].get(slot):
                        raise Hazard("S slot overwritten while the epilogue reads it")
                    m["S"][slot] = step
                    B[f"sfull{slot}"].arrive()
            yield

    def split(w):
        # split warp w: its rows of A for every MMA step, k-block by k-block as the previous
        # step's products release it; warp 0 refills a stage, once all four warps have read it
        # (pempty), with the P two MMA steps on
        if w == 0:
            for pc in range(min(stages, len(mma_steps))):
                load_p(pc)
        for pc, step in enumerate(mma_steps):
            st = pc % stages
            yield from wait(f"pfull{st}", pc // stages)
            m["Preading"][(st, w)] = True
            for b in range(4):
                if m["P"].get(st) != step:
                    raise Hazard(f"split warp {w} reads a stale P stage")
                yield
                if pc >= 1 and mistake != "a_without_empty":
                    yield from wait(f"aempty{b}", pc - 1)
                touches([("A", (b, w))], True, "split")
                m["A"][(b, w)] = step
                B[f"afull{b}"].arrive()
                yield
            m["Preading"][(st, w)] = False
            B[f"pempty{st}"].arrive()
            if w == 0:
                if mistake != "p_without_empty":
                    yield from wait(f"pempty{st}", pc // stages)
                load_p(pc + stages)

    def issuer(i):
        # issuer i: k-step i of every k-block (its three products) into its own accumulator
        # D_i; k-block b goes back once all four issuers' products on it have completed
        for pc, step in enumerate(mma_steps):
            if mistake != "mma_without_x":
                yield from wait("xfull", pc)
            for b in range(4):
                yield from wait(f"afull{b}", pc)
                queues[i].append(("mma", dict(step=step, b=b, i=i)))
                queues[i].append(("commit", f"aempty{b}"))
                yield
            queues[i].append(("commit", "dfull"))

    def pipe():
        # the tensor core: products of one issuer start and complete in issue order, those of
        # different issuers interleave freely; a commit fires once every product its issuer
        # issued before it has completed
        while True:
            moves = [("complete", i) for i in range(4) if inflight[i]]
            moves += [("head", i) for i in range(4) if queues[i]]
            if moves:
                kind, i = rnd.choice(moves)
                if kind == "complete":
                    op = inflight[i].pop(0)
                    for (name, b), v in rw(op)[1].items():
                        m[name][b] = v
                    done[i] += 1
                else:
                    what, x = queues[i].pop(0)
                    if what == "commit":
                        commits[i].append((started[i], x))
                    else:
                        reads, writes = rw(x)
                        for key, want in reads.items():
                            have = m[key[0]].get(key[1]) if isinstance(key, tuple) else m[key]
                            if have != want:
                                raise Hazard(f"MMA of step {x['step']} reads {key} holding {have}, needs {want}")
                        inflight[i].append(x)
                        started[i] += 1
                while commits[i] and commits[i][0][0] <= done[i]:
                    B[commits[i].pop(0)[1]].arrive()
            yield

    def bulk():
        # the bulk-store engine: reads each issued store's slot, in order, some time later
        while True:
            if stores and rnd.random() < 0.5:
                sl, step = stores[0]
                if m["S"].get(sl) != ("prefix", step):
                    raise Hazard(f"store of step {step} reads slot {sl} holding {m['S'].get(sl)}")
                stores.pop(0)
            yield

    def epilogue():
        # the epilogue warps; thread 0 also refills S slots: once a step's prefix store has
        # read its slot, the slot takes the S four steps on
        for sc in range(min(s_slots, len(steps))):
            load_s(sc)
        dc = 0
        for sc, (t, j) in enumerate(steps):
            if j == 0 and s0:
                touches(["X"], True, "X from S0")
                m["X"] = (t, "S0")
                B["xfull"].arrive()
                yield
            sl = sc % s_slots
            yield from wait(f"sfull{sl}", sc // s_slots)
            if m["S"].get(sl) != (t, j):
                raise Hazard(f"epilogue of step {(t, j)} reads S of step {m['S'].get(sl)}")
            m["Sreading"][sl] = True
            yield
            if (t, j) in mma_steps:
                yield from wait("dfull", dc)
                dc += 1
                for i in range(4):
                    if m["D"].get(i) != (t, j):
                        raise Hazard(f"epilogue of step {(t, j)} reads D_{i} of step {m['D'].get(i)}")
                touches([("D", i) for i in range(4)], False, "D read")
            yield
            if j + 1 < ns:
                touches(["X"], True, "X write")
                m["X"] = (t, j)
                B["xfull"].arrive()
            yield
            # prefix_j over S_j in the slot, then one bulk store of it; the previous step's
            # slot is refilled once its store has read it (at most one store still reading)
            m["S"][sl] = ("prefix", (t, j))
            stores.append((sl, (t, j)))
            if mistake != "slot_before_store_read":
                while len(stores) > 1:
                    yield
            if sc >= 1:
                m["Sreading"][(sc - 1) % s_slots] = False
                load_s(sc - 1 + s_slots)
            yield

    actors = {"tma": tma(), "pipe": pipe(), "epi": epilogue(), "bulk": bulk()}
    actors.update({f"mma{i}": issuer(i) for i in range(4)})
    actors.update({f"split{w}": split(w) for w in range(4)})
    speed = {k: rnd.choice((0.05, 1.0, 1.0, 4.0)) for k in actors}
    alive = set(actors)
    last, still = None, 0
    for _ in range(2000000):
        if alive <= {"pipe", "bulk", "tma"} and not any(queues) and not any(inflight) and not any(commits) \
                and not stores and not loads:
            return "ok"
        names = sorted(alive)
        name = rnd.choices(names, weights=[speed[k] for k in names])[0]
        try:
            next(actors[name])
        except StopIteration:
            alive.discard(name)
        state = tuple((k, b.done, b.arr) for k, b in sorted(B.items())) + \
            tuple(map(len, queues)) + tuple(map(len, inflight)) + tuple(done)
        still = still + 1 if state == last else 0
        last = state
        if still > 20000:
            return f"deadlock with {sorted(alive)} alive"
    return "no progress"


@pytest.mark.parametrize("ns", [1, 2, 3, 6])
@pytest.mark.parametrize("s0", [False, True])
@pytest.mark.parametrize("tiles", [1, 3])
def test_compose_cols_protocol_interleavings(ns, s0, tiles):
    for seed in range(8):
        assert _run(ns, s0, seed, tiles=tiles) == "ok"


@pytest.mark.parametrize("mistake", ["p_without_empty", "a_without_empty", "mma_without_x",
                                     "slot_before_store_read"])
def test_compose_cols_model_catches_planted_mistakes(mistake):
    hits = 0
    for seed in range(80):
        try:
            if mistake == "slot_before_store_read":   # single-segment tiles: S loads alone
                r = _run(1, False, seed, mistake, tiles=8)
            else:
                r = _run(6, True, seed, mistake, tiles=2)
        except Hazard:
            hits += 1
            break
        hits += r != "ok"
        if hits:
            break
    assert hits > 0


MODELLED_SOURCE = ("compose_cols.cu", "670a280bf16c")


def test_model_is_checked_against_the_current_kernel_source():
    from tests.helpers import kernel_code_hash
    name, recorded = MODELLED_SOURCE
    assert kernel_code_hash(name) == recorded, (
        f"{name} changed since this model was checked against it: re-check the model "
        f"against the new code, then record the new hash {kernel_code_hash(name)}")
