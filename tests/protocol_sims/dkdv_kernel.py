"""Barrier protocol of the dK / dV kernel (K/V-major, SS-form S^T and dP^T).

Per item (one K/V tile of one query head): the TMA producer loads K and V
into shared memory (KVFull; KVEmpty is committed by the MMA issuer after the
item's last product).  The query tiles that see the K/V tile come through two
stages of Q, dO and their LSE / Delta rows (QFull / QEmpty, the stage freed
by the commit after the tile's dK).  Per query tile i the MMA issuer runs
S^T(i) and dP^T(i) into TMEM, then dV(i) once the elementwise warps have
packed P^T over S^T (P), S^T(i+1), dK(i) once they have packed dS^T over
dP^T (DS), dP^T(i+1); MMAs execute in issue order, so S^T(i+1) follows the
dV(i) that reads P^T(i) and dP^T(i+1) follows the dK(i) that reads dS^T(i).
Each elementwise half (128 arrivals) reads and rewrites only its own columns
of S^T and dP^T.  At the end of the item the MMA issuer commits Acc, the
elementwise warps read dK / dV out and release them (AccFree).

mutation 1: S^T(i+1) issued before dV(i) has read P^T(i).
mutation 2: a Q / dO stage released after dV(i), before dK(i) has read Q.
mutation 3: the K / V buffer released before the item's last products.
"""
from .engine import Engine


def run(items, seed, mutation=0):
    """items: number of query tiles of each work item of one CTA."""
    e = Engine(seed)
    for n, c in [("KVFull", 1), ("KVEmpty", 1), ("S", 1), ("DP", 1), ("P", 256), ("DS", 256),
                 ("Acc", 1), ("AccFree", 256)]:
        e.bar(n, c)
    for st in range(2):
        e.bar(f"QFull{st}", 1)
        e.bar(f"QEmpty{st}", 1)

    def tma():
        qi = 0
        for k, nt in enumerate(items):
            yield ("wait", "KVEmpty", (k & 1) ^ 1)
            e.bars["KVFull"].arrive(1, 2)
            e.load("sK", ("K", k), "KVFull")
            e.load("sV", ("V", k), "KVFull")
            for _ in range(nt):
                st = qi & 1
                yield ("wait", f"QEmpty{st}", ((qi >> 1) & 1) ^ 1)
                e.bars[f"QFull{st}"].arrive(1, 3)
                e.load(f"sQ{st}", ("Q", qi), f"QFull{st}")
                e.load(f"sDO{st}", ("dO", qi), f"QFull{st}")
                e.load(f"sL{st}", ("L", qi), f"QFull{st}")
                qi += 1

    def mma():
        qi = p_ph = ds_ph = 0

        def issue_s(i, k):
            e.mma([("sK", ("K", k)), (f"sQ{i & 1}", ("Q", i))],
                  [("S0", ("S", i)), ("S1", ("S", i))])
            e.commit("S")

        def issue_dp(i, k):
            e.mma([("sV", ("V", k)), (f"sDO{i & 1}", ("dO", i))],
                  [("DP0", ("dP", i)), ("DP1", ("dP", i))])
            e.commit("DP")

        def issue_acc(acc, src, val, operand, i, k, zero):
            reads = [(f"{src}0", (val, i)), (f"{src}1", (val, i)), operand]
            if not zero:
                reads.append((acc, ("acc", k)))
            e.mma(reads, [(acc, ("acc", k))])

        for k, nt in enumerate(items):
            yield ("wait", "KVFull", k & 1)
            if mutation == 3:  # planted: K / V released at the start of the item
                e.commit("KVEmpty")
            if nt:
                yield ("wait", f"QFull{qi & 1}", (qi >> 1) & 1)
                issue_s(qi, k)
                issue_dp(qi, k)
            first = True
            for j in range(nt):
                st, nhave = qi & 1, j + 1 < nt
                yield ("wait", "P", p_ph)
                p_ph ^= 1
                if first:
                    yield ("wait", "AccFree", (k & 1) ^ 1)
                if nhave and mutation == 1:  # planted: S^T(i+1) ahead of dV(i)
                    yield ("wait", f"QFull{(qi + 1) & 1}", ((qi + 1) >> 1) & 1)
                    issue_s(qi + 1, k)
                issue_acc("DV", "S", "P", (f"sDO{st}", ("dO", qi)), qi, k, first)
                if mutation == 2:  # planted: the stage released before dK(i)
                    e.commit(f"QEmpty{st}")
                if nhave and mutation != 1:
                    yield ("wait", f"QFull{(qi + 1) & 1}", ((qi + 1) >> 1) & 1)
                    issue_s(qi + 1, k)
                yield ("wait", "DS", ds_ph)
                ds_ph ^= 1
                issue_acc("DK", "DP", "dS", (f"sQ{st}", ("Q", qi)), qi, k, first)
                if mutation != 2:
                    e.commit(f"QEmpty{st}")
                if nhave:
                    issue_dp(qi + 1, k)
                first = False
                qi += 1
            if nt == 0:
                yield ("wait", "AccFree", (k & 1) ^ 1)
            e.commit("Acc")
            if mutation != 3:
                e.commit("KVEmpty")

    def elementwise(h):
        qi = s_ph = dp_ph = 0
        for k, nt in enumerate(items):
            for _ in range(nt):
                st = qi & 1
                yield ("wait", f"QFull{st}", (qi >> 1) & 1)
                yield ("wait", "S", s_ph)
                s_ph ^= 1
                e.expect(f"S{h}", ("S", qi))
                e.expect(f"sL{st}", ("L", qi))
                yield ("step",)
                e.expect(f"S{h}", ("S", qi))
                e.mem[f"S{h}"] = ("P", qi)
                e.bars["P"].arrive(128)
                yield ("wait", "DP", dp_ph)
                dp_ph ^= 1
                e.expect(f"DP{h}", ("dP", qi))
                e.expect(f"sL{st}", ("L", qi))
                yield ("step",)
                e.expect(f"DP{h}", ("dP", qi))
                e.mem[f"DP{h}"] = ("dS", qi)
                e.bars["DS"].arrive(128)
                qi += 1
            yield ("wait", "Acc", k & 1)
            if nt:
                e.expect("DV", ("acc", k))
                e.expect("DK", ("acc", k))
            yield ("step",)
            e.bars["AccFree"].arrive(128)

    e.roles = {"tma": tma(), "mma": mma(), "ew0": elementwise(0), "ew1": elementwise(1)}
    e.run()
