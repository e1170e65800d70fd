"""Host model of the synchronisation protocol of the dense compose kernel (csrc/compose_tc.cu).

The kernel's producer warp (TMA of the P and S tiles), MMA issuer, the tensor pipe that runs the
issued products in order, and the epilogue warps (taken together as one agent: they arrive and
wait in the same order) are run here as coroutines under random interleavings, with the kernel's
barriers as phase counters. Each run checks that

- no interleaving deadlocks;
- no wait can alias a phase two ahead (the kernel waits on parities);
- no data is overwritten while a reader still needs it: the two D accumulators, the two halves
  of the A operand, the two P stages (split in place), the two low-part slots and the S tile.

The epilogue threads' own max-reduction of a transition unit's step (an mbarrier that only
they arrive at and wait on, with three value slots) orders nothing between agents, so the
model, which takes them as one agent, has no step for it.

The model follows the kernel's loop structure step by step (units, then segments; the P split of
step j + 1 interleaved with the two halves of step j's epilogue). It runs on the CPU only.
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


def _run(U, NS, has_s0, p_total, seed, mistake=None):
    """One random interleaving; returns "ok" or a deadlock description, raises Hazard."""
    rnd = random.Random(seed)
    units = range(2 * U if p_total else U)
    B = {n: _Bar() for n in ("p_full0", "p_full1", "p_empty0", "p_empty1", "lo_full0", "lo_full1",
                             "lo_empty0", "lo_empty1", "s_full", "s_empty", "a_full0", "a_full1",
                             "d_full")}
    st = dict(P={0: None, 1: None}, lo={0: None, 1: None}, A={b: None for b in range(4)},
              reading_D=None, reading_S=False, pend=[])
    n_buf = 1 if mistake == "one_d_buffer" else 2

    def wait(name, phase):
        b = B[name]
        if b.done > phase + 1:
            raise Hazard(f"parity alias on {name}")
        while b.done <= phase:
            yield

    def pending(field, value):   # a product still queued whose field (a tuple index) is value
        return any(op[0] == "mma" and op[field] == value for op in st["pend"])

    def producer():
        pc = sc = 0
        for ux in units:
            tr = ux >= U
            for j in range(NS):
                if j > 0 or (has_s0 and not tr):
                    s, use = pc & 1, pc >> 1
                    if use >= 1:
                        yield from wait(f"p_empty{s}", use - 1)
                    if pending(2, s):
                        raise Hazard("P stage reloaded under a pending product")
                    st["P"][s] = ("raw", pc)
                    B[f"p_full{s}"].arrive()
                    pc += 1
                if tr and j > 0:
                    continue
                if sc >= 1:
                    yield from wait("s_empty", sc - 1)
                if st["reading_S"]:
                    raise Hazard("S tile reloaded while read")
                B["s_full"].arrive()
                sc += 1
                yield

    def mma():
        pc = lb = ac = 0
        for ux in units:
            tr = ux >= U
            for j in range(NS):
                if not (j > 0 or (has_s0 and not tr)):
                    continue
                s, dbuf = pc & 1, pc % n_buf
                for b in range(4):
                    if b % 2 == 0:
                        yield from wait(f"a_full{b >> 1}", ac)
                    slot, use = lb & 1, lb >> 1
                    if mistake != "no_lo_wait":
                        yield from wait(f"lo_full{slot}", use)
                    st["pend"].append(("mma", pc, s, slot, b, dbuf))
                    st["pend"].append(("commit", f"lo_empty{slot}"))
                    lb += 1
                    yield
                ac += 1
                st["pend"].append(("commit", f"p_empty{s}"))
                st["pend"].append(("commit", "d_full"))
                pc += 1

    def pipe():
        while True:
            if st["pend"]:
                op = st["pend"].pop(0)
                if op[0] == "commit":
                    B[op[1]].arrive()
                else:
                    _, step, s, slot, b, dbuf = op
                    if st["reading_D"] == dbuf:
                        raise Hazard("product writes a D buffer the epilogue is reading")
                    if st["A"][b] != step:
                        raise Hazard("product reads a stale A block")
                    if st["lo"][slot] != (step, b):
                        raise Hazard("product reads a stale low-part slot")
                    if st["P"][s] != ("split", step):
                        raise Hazard("product reads an unsplit P stage")
            yield

    def epilogue():
        E = dict(pc=0, sc=0, lb=0, dc=0)

        def split(b0, b1):
            s, use = E["pc"] & 1, E["pc"] >> 1
            if b0 == 0:
                yield from wait(f"p_full{s}", use)
                st["P"][s] = ("split", E["pc"])
            for b in range(b0, b1):
                slot, luse = E["lb"] & 1, E["lb"] >> 1
                if luse >= 1:
                    yield from wait(f"lo_empty{slot}", luse - 1)
                if pending(3, slot):
                    raise Hazard("low-part slot rewritten under a pending product")
                st["lo"][slot] = (E["pc"], b)
                B[f"lo_full{slot}"].arrive()
                E["lb"] += 1
                yield
            if b1 == 4:
                E["pc"] += 1

        steps = 0   # products issued so far: the A version the next product reads
        for ux in units:
            tr = ux >= U
            if has_s0 and not tr:
                for b in range(4):
                    if pending(4, b):
                        raise Hazard("A written under a pending product")
                    st["A"][b] = steps
                B["a_full0"].arrive()
                B["a_full1"].arrive()
            split_ahead = False
            for j in range(NS):
                if j > 0 or (has_s0 and not tr):
                    if not split_ahead:
                        yield from split(0, 4)
                    dbuf = E["dc"] % n_buf
                    yield from wait("d_full", E["dc"])
                    E["dc"] += 1
                    st["reading_D"] = dbuf
                    steps += 1
                has_s = not (tr and j > 0)
                if has_s:
                    yield from wait("s_full", E["sc"])
                    E["sc"] += 1
                    st["reading_S"] = True
                nxt = j + 1 < NS
                for part in range(2):
                    yield
                    if nxt:
                        for b in (2 * part, 2 * part + 1):
                            if pending(4, b):
                                raise Hazard("A block written under a pending product")
                            st["A"][b] = steps
                    if part == 1:
                        st["reading_D"] = None
                        if has_s:
                            st["reading_S"] = False
                            B["s_empty"].arrive()
                    if nxt:
                        B[f"a_full{part}"].arrive()
                        yield from split(2 * part, 2 * part + 2)
                split_ahead = nxt

    actors = {"producer": producer(), "mma": mma(), "pipe": pipe(), "epilogue": epilogue()}
    alive = set(actors)
    last, still = None, 0
    for _ in range(100000):
        if alive <= {"pipe"} and not st["pend"]:
            return "ok"
        name = rnd.choice(sorted(alive))
        try:
            next(actors[name])
        except StopIteration:
            alive.discard(name)
        state = tuple((k, b.done, b.arr) for k, b in sorted(B.items())) + (len(st["pend"]),)
        still = still + 1 if state == last else 0
        last = state
        if still > 2000:
            return f"deadlock with {sorted(alive)} alive"
    return "no progress"


CASES = [(U, NS, s0, pt) for U in (1, 2) for NS in (1, 2, 3, 5) for s0 in (False, True)
         for pt in (False, True)]


@pytest.mark.parametrize("U,NS,has_s0,p_total", CASES)
def test_compose_protocol_interleavings(U, NS, has_s0, p_total):
    for seed in range(12):
        assert _run(U, NS, has_s0, p_total, seed) == "ok"


@pytest.mark.parametrize("mistake,expect", [
    ("one_d_buffer", ("D buffer",)),
    ("no_lo_wait", ("low-part", "unsplit P", "P stage")),
])
def test_compose_protocol_model_catches_planted_mistakes(mistake, expect):
    """The model is sharp enough to see a broken protocol: one D buffer instead of two, or
    products that do not wait for their low-part slot (then they read a slot, or a P stage,
    that the split has not written yet)."""
    hits = 0
    for seed in range(40):
        try:
            _run(1, 3, True, False, seed, mistake)
        except Hazard as h:
            assert any(e in str(h) for e in expect), str(h)
            hits += 1
    assert hits > 0


# The kernel source this model was last checked against (code only; comments do not count).
MODELLED_SOURCE = ("compose_tc.cu", "1fc5103a21f7")


def test_model_is_checked_against_the_current_kernel_source():
    from tests.helpers import kernel_code_hash
    name, recorded = MODELLED_SOURCE
    assert kernel_code_hash(name) == recorded, (
        f"{name} changed since this model was checked against it: re-check the model "
        f"against the new code, then record the new hash {kernel_code_hash(name)}")
