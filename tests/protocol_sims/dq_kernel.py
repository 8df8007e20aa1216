"""Barrier protocol of the dQ kernel (query-major, TS-form S and dP).

Per item (one query tile): the TMA producer loads Q and dO into shared memory
(QFull), then each K/V tile j into rings of three K and two V slots; the
elementwise warps (two halves, 128 arrivals each) copy Q / dO into TMEM
(QT) and release the shared-memory copy (QEmpty); the MMA issuer runs
S(j+1) after SFree(j), dQ(j) after DS(j) (reading the dS packed over dP(j)),
then dP(j+1) over the same dP buffer; each elementwise half reads S, then
dP, and rewrites only the dP columns it read itself with dS.

mutation 1: dP(j+1) issued before dQ(j) has read dS(j).
mutation 2: the shared-memory Q / dO released before the copy into TMEM.
mutation 3: the MMA issuer does not wait for the copy into TMEM.
"""
from .engine import Engine

KS, VS = 3, 2


def run(items, seed, mutation=0):
    """items: number of K/V tiles of each work item of one CTA."""
    e = Engine(seed)
    for n, c in [("QFull", 1), ("QEmpty", 256), ("S", 1), ("SFree", 256), ("DP", 1),
                 ("DS", 256), ("QT", 256), ("Acc", 1), ("AccFree", 256)]:
        e.bar(n, c)
    for i in range(KS):
        e.bar(f"KFull{i}", 1)
        e.bar(f"KEmpty{i}", 1)
    for i in range(VS):
        e.bar(f"VFull{i}", 1)
        e.bar(f"VEmpty{i}", 1)

    def tma():
        tj = 0
        for k, nt in enumerate(items):
            yield ("wait", "QEmpty", (k & 1) ^ 1)
            e.bars["QFull"].arrive(1, 2)
            e.load("sQ", ("Q", k), "QFull")
            e.load("sDO", ("dO", k), "QFull")
            for _ in range(nt):
                ks, vs = tj % KS, tj % VS
                yield ("wait", f"KEmpty{ks}", ((tj // KS) & 1) ^ 1)
                e.bars[f"KFull{ks}"].arrive(1, 1)
                e.load(f"K{ks}", ("K", tj), f"KFull{ks}")
                yield ("wait", f"VEmpty{vs}", ((tj // VS) & 1) ^ 1)
                e.bars[f"VFull{vs}"].arrive(1, 1)
                e.load(f"V{vs}", ("V", tj), f"VFull{vs}")
                tj += 1

    def mma():
        kj = sf_ph = ds_ph = 0

        def issue_s(j, k):
            e.mma([("QT", ("Q", k)), (f"K{j % KS}", ("K", j))], [("S", ("S", j))])
            e.commit("S")

        def issue_dp(j, k):
            e.mma([("DOT", ("dO", k)), (f"V{j % VS}", ("V", j))],
                  [("DP0", ("dP", j)), ("DP1", ("dP", j))])
            e.commit("DP")
            e.commit(f"VEmpty{j % VS}")

        def wait_k(j):
            return ("wait", f"KFull{j % KS}", (j // KS) & 1)

        def wait_v(j):
            return ("wait", f"VFull{j % VS}", (j // VS) & 1)

        for k, nt in enumerate(items):
            if mutation != 3:
                yield ("wait", "QT", k & 1)
            if nt:
                yield wait_k(kj)
                issue_s(kj, k)
                yield wait_v(kj)
                issue_dp(kj, k)
            first = True
            for j in range(nt):
                nhave = j + 1 < nt
                if nhave:
                    yield wait_k(kj + 1)
                    yield ("wait", "SFree", sf_ph)
                    sf_ph ^= 1
                    issue_s(kj + 1, k)
                    if mutation == 1:
                        yield wait_v(kj + 1)
                        issue_dp(kj + 1, k)
                yield ("wait", "DS", ds_ph)
                ds_ph ^= 1
                if first:
                    yield ("wait", "AccFree", (k & 1) ^ 1)
                reads = [("DP0", ("dS", kj)), ("DP1", ("dS", kj)), (f"K{kj % KS}", ("K", kj))]
                if not first:
                    reads.append(("DQ", ("acc", k)))
                e.mma(reads, [("DQ", ("acc", k))])
                e.commit(f"KEmpty{kj % KS}")
                if nhave and mutation != 1:
                    yield wait_v(kj + 1)
                    issue_dp(kj + 1, k)
                first = False
                kj += 1
            if nt == 0:
                yield ("wait", "AccFree", (k & 1) ^ 1)
            else:
                yield ("wait", "SFree", sf_ph)
                sf_ph ^= 1
            e.commit("Acc")

    def elementwise(h):
        kj = s_ph = dp_ph = 0
        src, dst, name = ("sQ", "QT", "Q") if h == 0 else ("sDO", "DOT", "dO")
        for k, nt in enumerate(items):
            yield ("wait", "QFull", k & 1)
            if mutation == 2:
                e.bars["QEmpty"].arrive(128)
                yield ("step",)
            e.expect(src, (name, k))
            yield ("step",)
            e.expect(src, (name, k))
            e.mem[dst] = (name, k)
            e.bars["QT"].arrive(128)
            if mutation != 2:
                e.bars["QEmpty"].arrive(128)
            for _ in range(nt):
                yield ("wait", "S", s_ph)
                s_ph ^= 1
                e.expect("S", ("S", kj))
                yield ("step",)
                e.bars["SFree"].arrive(128)
                yield ("wait", "DP", dp_ph)
                dp_ph ^= 1
                e.expect(f"DP{h}", ("dP", kj))
                yield ("step",)
                e.expect(f"DP{h}", ("dP", kj))
                e.mem[f"DP{h}"] = ("dS", kj)
                e.bars["DS"].arrive(128)
                kj += 1
            yield ("wait", "Acc", k & 1)
            if nt:
                e.expect("DQ", ("acc", k))
            yield ("step",)
            e.bars["AccFree"].arrive(128)

    e.roles = {"tma": tma(), "mma": mma(), "ew0": elementwise(0), "ew1": elementwise(1)}
    e.run()
