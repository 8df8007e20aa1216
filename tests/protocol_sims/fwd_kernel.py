"""Barrier protocol of the forward kernel (two query tiles per item).

Per item (a pair of 128-row query tiles): the TMA producer loads both Q
tiles (QFull; QEmpty is committed after the item's last product), then each
K/V tile j into a ring of five slots, K(j) and V(j) in consecutive entries
(Full / Empty per slot).  A K/V tile may serve one or both query tiles (its
use mask).  The MMA issuer runs S_i(j) for each query tile i that uses tile
j and releases K(j)'s slot behind them; per tile j it then waits for V(j),
and for each query tile i runs P V_i(j) once softmax warpgroup i has
packed P over S_i (P_i), then S_i(j+1) into the same columns; it releases
V(j)'s slot, and K(j+1)'s, behind them.  At the end of the item it commits
O_i for each query tile that had a product, and QEmpty.  Softmax warpgroup
i (128 arrivals) reads S_i, may rescale O_i in TMEM (between P V_i(j-1),
which the S_i barrier covers, and P V_i(j), issued after its P_i arrival),
and writes P over S_i; at the end of an item with at least one tile it
waits for O_i and reads O out.  The O tags count the products, so a
rescale or a read-out that overlaps a product fails.

mutation 1: O_0 and O_1 committed at the end of every item, whichever
            query tiles had products (a warpgroup with none does not wait).
mutation 2: P V_i(j) issued without waiting for P_i.
mutation 3: K(j)'s slot released before its S products are issued.
"""
from .engine import Engine

SLOTS = 5


def run(items, seed, mutation=0):
    """items: per work item, the use mask of each K/V tile (1: query tile 0,
    2: query tile 1, 3: both)."""
    e = Engine(seed)
    for n, c in [("QFull", 1), ("QEmpty", 1)]:
        e.bar(n, c)
    for i in range(2):
        e.bar(f"S{i}", 1)
        e.bar(f"P{i}", 128)
        e.bar(f"O{i}", 1)
    for s in range(SLOTS):
        e.bar(f"Full{s}", 1)
        e.bar(f"Empty{s}", 1)
    products = {}  # (item, query tile) -> P V products issued so far

    def tma():
        seq = 0
        for k, tiles in enumerate(items):
            yield ("wait", "QEmpty", (k & 1) ^ 1)
            e.bars["QFull"].arrive(1, 2)
            e.load("sQ0", ("Q", k, 0), "QFull")
            e.load("sQ1", ("Q", k, 1), "QFull")
            for j in range(len(tiles)):
                for which in ("K", "V"):
                    s = seq % SLOTS
                    yield ("wait", f"Empty{s}", ((seq // SLOTS) & 1) ^ 1)
                    e.bars[f"Full{s}"].arrive(1, 1)
                    e.load(f"slot{s}", (which, k, j), f"Full{s}")
                    seq += 1

    def mma():
        kv_it = 0
        p_ph = [0, 0]

        def issue_s(i, k, j, n):
            e.mma([(f"sQ{i}", ("Q", k, i)), (f"slot{n % SLOTS}", ("K", k, j))],
                  [(f"S{i}", ("S", k, i, j))])
            e.commit(f"S{i}")

        for k, tiles in enumerate(items):
            yield ("wait", "QFull", k & 1)
            if not tiles:
                e.commit("QEmpty")
                continue
            kn = 2 * kv_it
            yield ("wait", f"Full{kn % SLOTS}", (kn // SLOTS) & 1)
            if mutation == 3:  # planted: K(0)'s slot released before its S products
                e.commit(f"Empty{kn % SLOTS}")
            for i in range(2):
                if tiles[0] >> i & 1:
                    issue_s(i, k, 0, kn)
            if mutation != 3:
                e.commit(f"Empty{kn % SLOTS}")
            acc = [0, 0]
            for j, fl in enumerate(tiles):
                have_next = j + 1 < len(tiles)
                vn, nkn = 2 * kv_it + 1, 2 * kv_it + 2
                yield ("wait", f"Full{vn % SLOTS}", (vn // SLOTS) & 1)
                k_ready = False
                for i in range(2):
                    if fl >> i & 1:
                        if mutation != 2:
                            yield ("wait", f"P{i}", p_ph[i])
                            p_ph[i] ^= 1
                        c = products.get((k, i), 0)
                        reads = [(f"S{i}", ("P", k, i, j)), (f"slot{vn % SLOTS}", ("V", k, j))]
                        if acc[i]:
                            reads.append((f"O{i}", ("O", k, i, c)))
                        e.mma(reads, [(f"O{i}", ("O", k, i, c + 1))])
                        products[(k, i)] = c + 1
                        acc[i] = 1
                    if have_next and tiles[j + 1] >> i & 1:
                        if not k_ready:
                            yield ("wait", f"Full{nkn % SLOTS}", (nkn // SLOTS) & 1)
                            k_ready = True
                        issue_s(i, k, j + 1, nkn)
                e.commit(f"Empty{vn % SLOTS}")
                if have_next:
                    e.commit(f"Empty{nkn % SLOTS}")
                kv_it += 1
            for i in range(2):
                if acc[i] or mutation == 1:
                    e.commit(f"O{i}")
            e.commit("QEmpty")

    def softmax(ti):
        s_ph = o_ph = 0
        for k, tiles in enumerate(items):
            nt = 0
            for j, fl in enumerate(tiles):
                if not fl >> ti & 1:
                    continue
                yield ("wait", f"S{ti}", s_ph)
                s_ph ^= 1
                e.expect(f"S{ti}", ("S", k, ti, j))
                if nt > 0:  # rescale O in TMEM: after P V(j-1), before P V(j)
                    e.expect(f"O{ti}", ("O", k, ti, nt))
                    yield ("step",)
                    e.expect(f"O{ti}", ("O", k, ti, nt))
                yield ("step",)
                e.expect(f"S{ti}", ("S", k, ti, j))
                e.mem[f"S{ti}"] = ("P", k, ti, j)
                e.bars[f"P{ti}"].arrive(128)
                nt += 1
            if nt == 0:
                continue
            yield ("wait", f"O{ti}", o_ph)
            o_ph ^= 1
            e.expect(f"O{ti}", ("O", k, ti, nt))
            yield ("step",)

    e.roles = {"tma": tma(), "mma": mma(), "sm0": softmax(0), "sm1": softmax(1)}
    e.run()
