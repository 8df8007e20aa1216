"""Barrier protocol of the one-pass backward kernel (K/V-major; dK, dV and dQ
from one walk, dQ added by bulk reductions).

Per item (one K/V tile of one query head) the CTA walks its query tiles
(Q / dO / LSE stages double-buffered).  TMEM columns: X (S^T, then P^T
packed over it), Y (dP^T, then dS^T packed over it, then dQ^T), dV, dK.  The
shared-memory buffer DS holds dS^T for the dQ^T product, then the drain's
float32 staging of dQ^T (two 16 KB stage slots) that bulk reductions read.
MMA order per tile: dV, dK, dQ^T, S(next), then dP(next) once the drain has
read dQ^T out of Y.  The elementwise and drain halves are modelled as two
agents each (128 arrivals; the drain's leader issues the reductions).

mutation 1: the MMA issuer does not wait for the drain (YFree) before dP(next).
mutation 2: the elementwise warps do not wait for the staging buffer (DSFree)
            before writing dS^T.
mutation 3: the drain does not wait for a stage slot's reduction (StageFree)
            before refilling it.
"""
from .engine import Engine


def run(items, seed, mutation=0):
    """items: number of query tiles of each work item of one CTA."""
    e = Engine(seed)
    for n, c in [("KVFull", 1), ("KVEmpty", 1), ("QFull0", 1), ("QFull1", 1), ("QEmpty0", 1),
                 ("QEmpty1", 1), ("S", 1), ("DP", 1), ("P", 256), ("DS", 256), ("DQ", 1),
                 ("YFree", 128), ("DSFree", 1), ("StageFull0", 128), ("StageFull1", 128),
                 ("StageFree0", 1), ("StageFree1", 1), ("Acc", 1), ("AccFree", 256)]:
        e.bar(n, c)
    group = [0]

    def tma():
        qi = 0
        for k, nt in enumerate(items):
            yield ("wait", "KVEmpty", (k & 1) ^ 1)
            e.bars["KVFull"].arrive(1, 2)
            e.load("K", k, "KVFull")
            e.load("V", k, "KVFull")
            for _ in range(nt):
                st = qi & 1
                yield ("wait", f"QEmpty{st}", ((qi >> 1) & 1) ^ 1)
                e.bars[f"QFull{st}"].arrive(1, 3)
                for r in ("Q", "DO", "LSE"):
                    e.load(f"{r}{st}", qi, f"QFull{st}")
                qi += 1

    def mma():
        qi = p_ph = ds_ph = 0

        def s_and_dp(q, st):
            e.mma([("K", k_cur[0]), (f"Q{st}", q)], [("X0", ("S", q)), ("X1", ("S", q))])
            e.commit("S")
            if mutation != 1:
                yield ("wait", "YFree", (q & 1) ^ 1)
            e.mma([("V", k_cur[0]), (f"DO{st}", q)], [("Y0", ("dP", q)), ("Y1", ("dP", q))])
            e.commit("DP")

        k_cur = [0]
        for k, nt in enumerate(items):
            k_cur[0] = k
            yield ("wait", "KVFull", k & 1)
            if nt:
                yield ("wait", f"QFull{qi & 1}", (qi >> 1) & 1)
                yield from s_and_dp(qi, qi & 1)
            for j in range(nt):
                st, nst = qi & 1, (qi + 1) & 1
                first = j == 0
                yield ("wait", "P", p_ph)
                p_ph ^= 1
                if first:
                    yield ("wait", "AccFree", (k & 1) ^ 1)
                e.mma([("X0", ("P", qi)), ("X1", ("P", qi)), (f"DO{st}", qi)] +
                      ([] if first else [("dV", ("acc", k))]), [("dV", ("acc", k))])
                yield ("wait", "DS", ds_ph)
                ds_ph ^= 1
                e.mma([("Y0", ("dSt", qi)), ("Y1", ("dSt", qi)), (f"Q{st}", qi)] +
                      ([] if first else [("dK", ("acc", k))]), [("dK", ("acc", k))])
                e.commit(f"QEmpty{st}")
                e.mma([("K", k), ("DS0", ("dS", qi)), ("DS1", ("dS", qi))],
                      [("Y0", ("dQ", qi)), ("Y1", ("dQ", qi))])
                e.commit("DQ")
                if j + 1 < nt:
                    yield ("wait", f"QFull{nst}", ((qi + 1) >> 1) & 1)
                    yield from s_and_dp(qi + 1, nst)
                qi += 1
            if nt == 0:
                yield ("wait", "AccFree", (k & 1) ^ 1)
            e.commit("Acc")
            e.commit("KVEmpty")

    def elementwise(h):
        qi = s_ph = dp_ph = 0
        for k, nt in enumerate(items):
            for _ in range(nt):
                st = qi & 1
                yield ("wait", f"QFull{st}", (qi >> 1) & 1)
                yield ("wait", "S", s_ph)
                s_ph ^= 1
                e.expect(f"X{h}", ("S", qi))
                e.expect(f"LSE{st}", qi)
                yield ("step",)
                e.mem[f"X{h}"] = ("P", qi)
                e.bars["P"].arrive(128)
                yield ("wait", "DP", dp_ph)
                dp_ph ^= 1
                e.expect(f"Y{h}", ("dP", qi))
                e.expect(f"LSE{st}", qi)
                yield ("step",)
                if mutation != 2:
                    yield ("wait", "DSFree", (qi & 1) ^ 1)
                e.mem[f"DS{h}"] = ("dS", qi)
                e.mem[f"Y{h}"] = ("dSt", qi)
                e.bars["DS"].arrive(128)
                qi += 1
            yield ("wait", "Acc", k & 1)
            if nt:
                e.expect("dK", ("acc", k))
                e.expect("dV", ("acc", k))
            yield ("step",)
            e.bars["AccFree"].arrive(128)

    def reduce(slot, tag):
        group[0] += 1
        e.reduces.append((slot, tag, group[0]))
        return group[0]

    def drain(leader):
        qi = 0
        n = 1 if leader else 127
        for k, nt in enumerate(items):
            for _ in range(nt):
                yield ("wait", "DQ", qi & 1)
                e.expect("Y0", ("dQ", qi))
                e.expect("Y1", ("dQ", qi))
                for s in range(2):
                    if leader:
                        e.mem[f"DS{s}"] = ("st", qi, s)
                    e.bars[f"StageFull{s}"].arrive(n)
                yield ("step",)
                e.expect("Y0", ("dQ", qi))
                e.bars["YFree"].arrive(n)
                if leader:
                    gids = []
                    for s in range(2):
                        yield ("wait", f"StageFull{s}", 0)
                        gids.append(reduce(f"DS{s}", ("st", qi, s)))
                    yield ("until", lambda g=gids[0]: g in e.read_done)
                    e.bars["StageFree0"].arrive(1)
                    yield ("until", lambda g=gids[1]: g in e.read_done)
                    e.bars["StageFree1"].arrive(1)
                for s in range(2):
                    if mutation != 3:
                        yield ("wait", f"StageFree{s}", qi & 1)
                    if leader:
                        e.mem[f"DS{s}"] = ("st", qi, s + 2)
                    e.bars[f"StageFull{s}"].arrive(n)
                if leader:
                    gids = []
                    for s in range(2):
                        yield ("wait", f"StageFull{s}", 1)
                        gids.append(reduce(f"DS{s}", ("st", qi, s + 2)))
                    yield ("until", lambda gs=tuple(gids): all(g in e.read_done for g in gs))
                    e.bars["DSFree"].arrive(1)
                qi += 1

    e.roles = {"tma": tma(), "mma": mma(), "ew0": elementwise(0), "ew1": elementwise(1),
               "drain_leader": drain(True), "drain_rest": drain(False)}
    e.run()
