"""Host model of the synchronisation protocol of the GDN / DeltaNet chain kernel
(csrc/build_gdn_tc.cu), one (segment, value head) unit.

Roles, as in the kernel: the TMA warp (k chunks into a 3-slot ring, {v chunk, M2 record} into
another), the two MMA issuers (the S~ half: W, U, d_S, f_S; the P half: d_P, f_P), the operand
warps (gates, M1 = M2 scaled, the read-out of W into the -W^T operand), and the conversion warps
of each half (bf16 copies of Z and of D in TMEM). Each group of warps that arrives and waits
together is one agent. The KDA instance (kda=True) is the same protocol with four gate slots,
each with its own barrier, that both halves read (the Z pass of chunk c rescales the state per key
row with the slot of chunk c - 1, the outputs with that of the last chunk), no M1 (U reads the
record), and a state write in both Z passes. Issued MMAs complete in issue order per issuer, in any interleaving
between the two issuers; a commit fires when its issuer's earlier MMAs have completed.

Every run checks for deadlock, for parity aliasing (the kernel waits on parities), and that each
buffer is read in the version its reader needs and never overwritten under a pending reader:
TMEM (Z and D of both halves, the bf16 Z copies, whose S~ columns also hold the W accumulator),
the k and {v, M2} rings, the two -W^T operand slots, the two M1 slots and the two per-chunk slots
of gate values. It runs on the CPU only.
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


def _run(nch, seed, mistake=None, out=False, kda=False):
    """One unit of nch chunks. out: the outputs instance of the kernel, whose P-half issuer
    computes the masked Q K^T of every chunk (Q by TMA into a two-slot ring) and whose P-half
    warps turn it into the bf16 operand of the intra-chunk product and read the outputs out;
    the S-half issuer adds Q S~ before d_S and the intra-chunk product after f_S."""
    rnd = random.Random(seed)
    KS = VS = 3
    SL = 4 if out or kda else 2   # per-chunk gate slots, as in the kernel
    if mistake == "kda_two_slots":
        SL = 2
    B = {}
    for s_ in range(4):
        B[f"gready{s_}"] = _Bar()   # KDA: one per gate slot
    for s in range(KS):
        B[f"kfull{s}"], B[f"kempty{s}"] = _Bar(), _Bar(2)
    for s in range(VS):
        B[f"vfull{s}"], B[f"vempty{s}"] = _Bar(), _Bar()
    for s in range(2):
        for n in ("m1ready", "zready", "dready", "wready"):
            B[f"{n}{s}"] = _Bar()   # one arrival per agent (128 threads in the kernel)
        for n in ("dfull", "zfull", "wfree"):
            B[f"{n}{s}"] = _Bar()
    B["wfull"] = _Bar()
    for s_ in range(2):
        B[f"qfull{s_}"], B[f"qempty{s_}"] = _Bar(), _Bar(2)   # qempty: Q S~ and Q K^T
        B[f"aqready{s_}"] = _Bar()
    for n_ in ("aqfull", "aqfree"):
        B[n_] = _Bar()
    for s_ in range(2):   # two output accumulators, by chunk parity
        B[f"ofull{s_}"], B[f"ofree{s_}"] = _Bar(), _Bar()
    # buffer contents (versions)
    m = dict(ZK0=None, ZK1=None, D0=None, D1=None, Z0=("Z", -1), Z1=("Z", -1), k={}, vr={},
             wop={}, m1={}, slot={}, w_read=set(), q={}, aq={}, AQ=None, O0=None, O1=None,
             slot_readers=set())
    queues = {0: [], 1: []}   # per issuer: pending MMAs and commits, in issue order

    def wait(name, phase):
        b = B[name]
        if b.done > phase + 1:
            raise Hazard(f"parity alias on {name}")
        while b.done <= phase:
            yield

    # ---------------------------------------------------------------- TMA warp
    def tma():
        for c in range(nch):
            ks, kuse = c % KS, c // KS
            if kuse >= 1:
                yield from wait(f"kempty{ks}", kuse - 1)
            touches_inflight([("k", ks)], True, "k load")
            m["k"][ks] = c
            B[f"kfull{ks}"].arrive()
            vs, vuse = c % VS, c // VS
            if vuse >= 1:
                yield from wait(f"vempty{vs}", vuse - 1)
            touches_inflight([("vr", vs)], True, "{v, M2} load")
            m["vr"][vs] = c
            B[f"vfull{vs}"].arrive()
            if out:
                qs, quse = c % 2, c // 2
                if quse >= 1 and mistake != "q_without_qempty":
                    yield from wait(f"qempty{qs}", quse - 1)
                touches_inflight([("q", qs)], True, "q load")
                m["q"][qs] = c
                B[f"qfull{qs}"].arrive()
            yield

    # ---------------------------------------------------------------- MMA issuers
    def issue(hf, op):
        queues[hf].append(("mma", op))

    def commit(hf, bar):
        queues[hf].append(("commit", bar))

    def issuer_s():
        if nch == 0:
            return
        yield from wait("kfull0", 0)
        yield from wait("vfull0", 0)
        issue(0, dict(kind="W", c=0, k=0, vr=0))
        commit(0, "wfull")
        yield from wait("m1ready0", 0)
        issue(0, dict(kind="U", c=0, vr=0, m1=0))
        commit(0, "vempty0")
        for c in range(nch):
            more = c + 1 < nch
            yield from wait(f"wready{c & 1}", c >> 1)
            yield from wait("zready0", c)
            if out:
                yield from wait(f"qfull{c % 2}", c // 2)
                if c >= 2 and mistake != "qs_without_ofree":
                    yield from wait(f"ofree{c & 1}", (c - 2) >> 1)
                issue(0, dict(kind="QS", c=c, q=c % 2))
            issue(0, dict(kind="dS", c=c, wop=c & 1))
            commit(0, "dfull0")
            if out:
                commit(0, f"qempty{c % 2}")
            yield
            if more:
                if mistake != "w_before_dS_done":
                    yield from wait("dfull0", c)
                yield from wait(f"kfull{(c + 1) % KS}", (c + 1) // KS)
                yield from wait(f"vfull{(c + 1) % VS}", (c + 1) // VS)
                issue(0, dict(kind="W", c=c + 1, k=(c + 1) % KS, vr=(c + 1) % VS))
                commit(0, "wfull")
            yield from wait("dready0", c)
            issue(0, dict(kind="fS", c=c, k=c % KS))
            if out:
                yield from wait(f"aqready{c & 1}", c >> 1)
                issue(0, dict(kind="intra", c=c, aq=c & 1))
            commit(0, "zfull0")
            commit(0, f"kempty{c % KS}")
            if out:
                commit(0, f"ofull{c & 1}")
            yield
            if more:
                yield from wait("zfull0", c)
                yield from wait(f"m1ready{(c + 1) & 1}", (c + 1) >> 1)
                issue(0, dict(kind="U", c=c + 1, vr=(c + 1) % VS, m1=(c + 1) & 1))
                commit(0, f"vempty{(c + 1) % VS}")

    def issuer_p():
        if out:   # Q K^T of every chunk into its TMEM accumulator
            for c in range(nch):
                yield from wait(f"qfull{c % 2}", c // 2)
                yield from wait(f"kfull{c % KS}", c // KS)
                if c >= 1 and mistake != "qk_without_aqfree":
                    yield from wait("aqfree", c - 1)
                issue(1, dict(kind="QK", c=c, q=c % 2, k=c % KS))
                commit(1, "aqfull")
                commit(1, f"qempty{c % 2}")
                commit(1, f"kempty{c % KS}")
                yield
            return
        for c in range(nch):
            yield from wait(f"wready{c & 1}", c >> 1)
            yield from wait("zready1", c)
            issue(1, dict(kind="dP", c=c, wop=c & 1))
            commit(1, "dfull1")
            commit(1, f"wfree{c & 1}")
            yield
            yield from wait("dready1", c)
            issue(1, dict(kind="fP", c=c, k=c % KS))
            commit(1, "zfull1")
            commit(1, f"kempty{c % KS}")

    # ---------------------------------------------------------------- tensor pipe
    # An MMA group reads its operands and writes its accumulator from its start to its
    # completion; groups of one issuer start and complete in issue order but may overlap (the
    # pipe is pipelined), and a commit fires once every earlier group of its issuer completed.
    inflight = {0: [], 1: []}
    started = {0: 0, 1: 0}      # groups started per issuer
    completed = {0: 0, 1: 0}    # groups completed per issuer
    commits = {0: [], 1: []}    # (groups that must complete first, barrier)

    def rw(op):
        kind, c = op["kind"], op["c"]
        if kind == "W":
            return {("k", op["k"]): c, ("vr", op["vr"]): c}, {"ZK0": ("W", c)}
        if kind == "U":
            if kda:   # B is the M2 record itself
                return {("vr", op["vr"]): c}, {"D0": ("U", c)}
            return {("vr", op["vr"]): c, ("m1", op["m1"]): c}, {"D0": ("U", c)}
        if kind == "dS":
            return {"ZK0": ("Z", c), ("wop", op["wop"]): c, "D0": ("U", c)}, {"D0": ("d", c)}
        ob = 0 if mistake == "one_output_buffer" else c & 1
        if kind == "QS":
            return {"ZK0": ("Z", c), ("q", op["q"]): c}, {f"O{ob}": ("QS", c)}
        if kind == "QK":
            return {("q", op["q"]): c, ("k", op["k"]): c}, {"AQ": ("AQ", c)}
        if kind == "intra":
            return {"D0": ("Dbf", c), ("aq", op["aq"]): c, f"O{ob}": ("QS", c)}, {f"O{ob}": ("O", c)}
        if kind == "dP":
            return {"ZK1": ("Z", c), ("wop", op["wop"]): c}, {"D1": ("d", c)}
        hf = 0 if kind == "fS" else 1
        return {f"D{hf}": ("Dbf", c), ("k", op["k"]): c, f"Z{hf}": ("Z", c - 1)}, {f"Z{hf}": ("Z", c)}

    def chained(x, y):
        """y may overlap x: the same accumulator, accumulated in issue order by one issuer."""
        return ((x["kind"] == "U" and y["kind"] == "dS") or (x["kind"] == "QS" and y["kind"] == "intra")) \
            and x["c"] == y["c"]

    def touches_inflight(keys, writing, who):
        for q in inflight.values():
            for x in q:
                xr, xw = rw(x)
                if any(k in xw for k in keys) or (writing and any(k in xr for k in keys)):
                    raise Hazard(f"{who} touches {keys} under the in-flight {x['kind']}({x['c']})")

    def start(hf, op):
        reads, writes = rw(op)
        for q in inflight.values():
            for x in q:
                if chained(x, op):
                    continue
                xr, xw = rw(x)
                if set(xw) & (set(reads) | set(writes)) or set(writes) & set(xr):
                    raise Hazard(f"{op['kind']}({op['c']}) overlaps the in-flight {x['kind']}({x['c']})")
        for key, want in reads.items():
            have = m.get(key) if isinstance(key, str) else m[key[0]].get(key[1])
            if have != want and not any(chained(x, op) and rw(x)[1].get(key) == want
                                        for x in inflight[hf]):
                raise Hazard(f"{op['kind']}({op['c']}) reads {key} holding {have}, needs {want}")
        inflight[hf].append(op)
        started[hf] += 1

    def fire(hf):
        while commits[hf] and commits[hf][0][0] <= completed[hf]:
            B[commits[hf].pop(0)[1]].arrive()

    def complete(hf):
        op = inflight[hf].pop(0)
        for key, val in rw(op)[1].items():
            m[key] = val
        completed[hf] += 1
        fire(hf)

    def pipe():
        while True:
            moves = []
            for hf in (0, 1):
                if inflight[hf]:
                    moves.append(("complete", hf))
                if queues[hf]:
                    moves.append(("head", hf))
            if moves:
                what, hf = rnd.choice(moves)
                if what == "complete":
                    complete(hf)
                else:
                    kind, payload = queues[hf].pop(0)
                    if kind == "commit":   # tracks the groups issued before it; does not stall
                        commits[hf].append((started[hf], payload))
                        fire(hf)
                    else:
                        start(hf, payload)
            yield

    # ---------------------------------------------------------------- operand warps
    def operand():
        for c in range(nch):
            if kda and any(r[0] == c % SL for r in m["slot_readers"]):
                raise Hazard("gate slot rewritten while a half reads it")
            m["slot"][c % SL] = c
            yield
            if kda:
                B[f"gready{c % SL}"].arrive()
                B[f"m1ready{c & 1}"].arrive()   # no M1: U reads the record
                yield
            else:
                yield from wait(f"vfull{c % VS}", c // VS)
                if m["vr"].get(c % VS) != c:
                    raise Hazard("M1 built from a stale record")
                touches_inflight([("m1", c & 1)], True, "M1 write")
                m["m1"][c & 1] = c
                B[f"m1ready{c & 1}"].arrive()
                yield
            yield from wait("wfull", c)
            if c >= 2 and mistake != "no_wfree" and not out:   # d_P's read of the slot
                yield from wait(f"wfree{c & 1}", (c - 2) >> 1)
            if m["ZK0"] != ("W", c):
                raise Hazard(f"W read-out finds {m['ZK0']}")
            touches_inflight(["ZK0"], False, "W read-out")
            touches_inflight([("wop", c & 1)], True, "-W^T write")
            m["wop"][c & 1] = c
            m["w_read"].add(c)
            B[f"wready{c & 1}"].arrive()

    # ---------------------------------------------------------------- conversion warps
    def read_slot(hf, c, what):
        # a half reads the gate slot of chunk c over some time
        m["slot_readers"].add((c % SL, hf))
        for _ in range(2):
            if m["slot"].get(c % SL) != c:
                raise Hazard(f"{what} reads the gate slot of another chunk")
            yield
        m["slot_readers"].discard((c % SL, hf))

    def conversion(hf):
        for c in range(nch):
            if c >= 1:
                yield from wait(f"zfull{hf}", c - 1)
            if kda:
                if c >= 1:
                    yield from wait(f"gready{(c - 1) % SL}", (c - 1) // SL)
                if hf == 0 and mistake != "no_wready_before_z":
                    yield from wait(f"wready{c & 1}", c >> 1)
                    if c >= 1 and c not in m["w_read"] and m["ZK0"] == ("W", c):
                        raise Hazard("Z copy written over W before its read-out")
                if c >= 1:
                    yield from read_slot(hf, c - 1, f"Z pass {hf}")
            elif hf == 0:
                yield from wait(f"m1ready{c & 1}", c >> 1)
                if mistake != "no_wready_before_z":
                    yield from wait(f"wready{c & 1}", c >> 1)
                if m["slot"].get(c % SL) != c:
                    raise Hazard("gate slot of another chunk")
                if c >= 1 and c not in m["w_read"] and m["ZK0"] == ("W", c):
                    raise Hazard("Z copy written over W before its read-out")
                if c >= 1 and m["ZK0"] != ("W", c) and any(x["kind"] == "W" for x in inflight[0]):
                    raise Hazard("Z copy written under the in-flight W")
            if m[f"Z{hf}"] != ("Z", c - 1):
                raise Hazard(f"Z conversion {hf} at chunk {c} reads {m[f'Z{hf}']}")
            touches_inflight([f"Z{hf}"], hf == 0 or kda, "Z conversion")   # a rescale writes Z
            touches_inflight([f"ZK{hf}"], True, "Z copy")
            m[f"ZK{hf}"] = ("Z", c)
            B[f"zready{hf}"].arrive()
            yield
            yield from wait(f"dfull{hf}", c)
            if m[f"D{hf}"] != ("d", c):
                raise Hazard(f"D conversion {hf} at chunk {c} reads {m[f'D{hf}']}")
            touches_inflight([f"D{hf}"], True, "D conversion")
            m[f"D{hf}"] = ("Dbf", c)
            B[f"dready{hf}"].arrive()
            yield
        if nch > 0:
            yield from wait(f"zfull{hf}", nch - 1)
            if m[f"Z{hf}"] != ("Z", nch - 1):
                raise Hazard("output reads a stale state")
            if kda:   # the last chunk's scaling (and lam)
                yield from wait(f"gready{(nch - 1) % SL}", (nch - 1) // SL)
                yield from read_slot(hf, nch - 1, "output")

    # ---------------------------------------------------------------- output warps (out)
    # the P-half warps of the outputs instance: the masked Q K^T into the bf16 B operand of the
    # intra-chunk product, then the outputs read out and scaled with the chunk's gate slot
    def outwarps():
        def prep_aq(c):
            yield from wait("aqfull", c)
            if m["AQ"] != ("AQ", c):
                raise Hazard(f"Q K^T read-out at chunk {c} finds {m['AQ']}")
            touches_inflight(["AQ"], False, "Q K^T read-out")
            B["aqfree"].arrive()
            yield
            touches_inflight([("aq", c & 1)], True, "masked Q K^T write")
            m["aq"][c & 1] = c
            B[f"aqready{c & 1}"].arrive()
            yield

        # the masked Q K^T of chunk c + 1 is prepared before the outputs of chunk c are read
        if nch > 0:
            yield from prep_aq(0)
        for c in range(nch):
            if c + 1 < nch:
                yield from prep_aq(c + 1)
            yield from wait(f"ofull{c & 1}", c >> 1)
            ob = 0 if mistake == "one_output_buffer" else c & 1
            if m[f"O{ob}"] != ("O", c):
                raise Hazard(f"output read-out at chunk {c} finds {m[f'O{ob}']}")
            touches_inflight([f"O{ob}"], False, "output read-out")
            # the outputs are scaled with the chunk's gate slot, read over some time, and the
            # accumulator freed after that
            for _ in range(2):
                if m["slot"].get(c % SL) != c:
                    raise Hazard("output scale read from the gate slot of another chunk")
                yield
            B[f"ofree{c & 1}"].arrive()

    if mistake == "three_gate_slots":
        SL = 3
    actors = {"tma": tma(), "s": issuer_s(), "p": issuer_p(), "pipe": pipe(), "op": operand(),
              "c0": conversion(0), "c1": outwarps() if out else conversion(1)}
    # per-run speeds: some runs starve one agent, so that the others run ahead as far as the
    # protocol lets them
    speed = {k: rnd.choice((0.05, 1.0, 1.0, 4.0)) for k in actors}
    alive = set(actors)
    last, still = None, 0
    for _ in range(400000):
        if alive <= {"pipe"} and not any(queues.values()) and not any(inflight.values()) and not any(commits.values()):
            return "ok"
        names = sorted(alive)
        name = rnd.choices(names, weights=[speed[k] for k in names])[0]
        try:
            next(actors[name])
        except StopIteration:
            alive.discard(name)
        state = tuple((k, b.done, b.arr) for k, b in sorted(B.items())) + (
            len(queues[0]), len(queues[1]), len(inflight[0]), len(inflight[1]), completed[0], completed[1])
        still = still + 1 if state == last else 0
        last = state
        if still > 20000:
            return f"deadlock with {sorted(alive)} alive"
    return "no progress"


@pytest.mark.parametrize("nch", [1, 2, 3, 4, 7])
def test_chain_protocol_interleavings(nch):
    for seed in range(25):
        assert _run(nch, seed) == "ok"


@pytest.mark.parametrize("nch", [1, 2, 3, 4, 7])
def test_outputs_instance_protocol_interleavings(nch):
    for seed in range(25):
        assert _run(nch, seed, out=True) == "ok"


@pytest.mark.parametrize("nch", [1, 2, 3, 4, 7, 9])
def test_kda_instance_protocol_interleavings(nch):
    for seed in range(25):
        assert _run(nch, seed, kda=True) == "ok"


@pytest.mark.parametrize("mistake", ["kda_two_slots", "no_wready_before_z", "w_before_dS_done"])
def test_kda_instance_model_catches_planted_mistakes(mistake):
    hits = 0
    for seed in range(80):
        try:
            r = _run(7, seed, mistake, kda=True)
        except Hazard:
            hits += 1
            continue
        hits += r != "ok"
    assert hits > 0


@pytest.mark.parametrize("mistake", ["q_without_qempty", "one_output_buffer", "qk_without_aqfree",
                                     "three_gate_slots"])
def test_outputs_instance_model_catches_planted_mistakes(mistake):
    hits = 0
    for seed in range(80):
        try:
            r = _run(6, seed, mistake, out=True)
        except Hazard:
            hits += 1
            continue
        hits += r != "ok"
    assert hits > 0


@pytest.mark.parametrize("mistake", ["no_wready_before_z", "no_wfree", "w_before_dS_done"])
def test_chain_protocol_model_catches_planted_mistakes(mistake):
    """Dropping any one of these waits lets some interleaving read or overwrite a buffer in the
    wrong version."""
    hits = 0
    for seed in range(60):
        try:
            r = _run(5, seed, mistake)
        except Hazard:
            hits += 1
            continue
        hits += r != "ok"
    assert hits > 0


# The kernel source this model was last checked against (code only; comments do not count).
MODELLED_SOURCE = ("build_gdn_tc.cu", "36b00f4cb906")


def test_model_is_checked_against_the_current_kernel_source():
    from tests.helpers import kernel_code_hash
    name, recorded = MODELLED_SOURCE
    assert kernel_code_hash(name) == recorded, (
        f"{name} changed since this model was checked against it: re-check the model "
        f"against the new code, then record the new hash {kernel_code_hash(name)}")
