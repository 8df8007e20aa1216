"""Pins of the CPU oracle against what the pages and mathematics fix.

Each ``pin_*`` function raises AssertionError when the oracle (optionally a
mutated build of it) disagrees with an independent fact:

* the cp=4 zigzag assignment printed in "Sequence Parallelism IV ...",
  section 3 (tests/golden/zigzag_cp4.txt);
* the contiguous shard coverage artifact of "Context Parallelism for
  Long-Context Training" (tests/golden/contiguous_shards_n8_p4.txt);
* a pure-Python brute force of the softmax definition at S <= 16;
* closed forms: constant V gives V, Q = 0 gives the running mean with
  LSE = ln(#keys), row 0 of a causal mask sees only key 0;
* "CP=1 equals the unsharded reference" and independence of the ring result
  from cp, layout and merge order ("Prove attention equivalence");
* central finite differences of the brute-force forward for dQ, dK, dV,
  plus the sum rules sum_j dV_j = sum_i dO_i and sum_j dK_j = 0;
* closed-form per-step tile and pair counts of the two layouts;
* document (packed-sequence) masks: brute force and finite differences with
  documents, one token per document (out = its own V, LSE = its own score),
  packed documents equal to each document run alone (so padding as a
  document of its own leaves real tokens untouched), one document equal to
  the plain mask, and the ring under documents equal to the definition;
* the all-gather schedule ("Context Parallelism in MegaDLMs", key-value
  communication patterns: each rank gathers all K/V, then attends in one
  pass; gradients summed over ranks and returned to the owners) equal to
  the definition, forward and backward, for every cp and layout, with and
  without documents;
* the Ulysses variant ("Sequence Parallelism IV", section 7: an all-to-all
  from sequence to head ownership, after which a rank has all tokens of a
  head slice): the all-to-all places rank r's head slice of every token in
  natural order, and the variant equals the definition, forward and
  backward, also when kv heads are fewer than ranks (shared kv heads);
* hierarchical context parallelism ("Context Parallelism in MegaDLMs",
  "Hierarchical Context Parallelism" and the a2a+p2p type of "Key-Value
  Communication Patterns"): the first-level all-to-all puts head slice a of
  level-two shard p on member a of group p, checked against the two levels'
  token lists written out independently, and the whole a2a+p2p schedule
  equals the definition, forward and backward, for level sizes [2, 2],
  [2, 4] and [4, 2];
* dK / dV on listed key rows from the definition's O and LSE: finite
  differences and the sum rules.

``test_mutations_are_caught`` compiles planted mistakes into the oracle and
checks that some pin fails for each.
"""
import math
import os

import numpy as np
import pytest

import oracle
from oracle import brute
from context_causal_attention_zigzag_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def small(B, H, Hkv, S, D, seed, dout=False):
    w = inputs.Workload("tiny", B, H, Hkv, S, D, 1, inputs.ZIGZAG, True,
                        inputs.torch.float32, seed=seed)
    q, k, v, do = inputs.generate(w, with_dout=dout)
    f = inputs.to_f32_numpy
    return f(q), f(k), f(v), (f(do) if dout else None)


def read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([int(x) for x in line.split()])
    return rows


# ----------------------------------------------------------------------------
# pins
# ----------------------------------------------------------------------------

def pin_zigzag_golden(m=0):
    rows = read_golden("zigzag_cp4.txt")
    cp = 4
    # Chunk length 1: the sharded order lists each rank's chunks in turn.
    order = oracle.shard_order(2 * cp, cp, oracle.ZIGZAG, mutation=m)
    expect = [c for r, a, b in rows for c in (a, b)]
    assert order.tolist() == expect, (order.tolist(), expect)
    # Chunk length 3: every chunk moves as a block.
    c = 3
    order = oracle.shard_order(2 * cp * c, cp, oracle.ZIGZAG, mutation=m)
    expect = [ch * c + o for r, a, b in rows for ch in (a, b) for o in range(c)]
    assert order.tolist() == expect


def pin_contiguous_golden(m=0):
    rows = read_golden("contiguous_shards_n8_p4.txt")
    order = oracle.shard_order(8, 4, oracle.CONTIGUOUS, mutation=m)
    flat = [t for r in rows for t in r[1:]]
    assert order.tolist() == flat == list(range(8))


def pin_coverage(m=0):
    for cp in (1, 2, 3, 4, 8, 16):
        for layout, per in ((oracle.ZIGZAG, 2), (oracle.CONTIGUOUS, 1)):
            for c in (1, 2, 5):
                S = cp * per * c
                order = oracle.shard_order(S, cp, layout, mutation=m)
                assert sorted(order.tolist()) == list(range(S))
                if layout == oracle.ZIGZAG and c == 1:
                    assign = brute.zigzag_assignment(cp)
                    assert order.tolist() == [x for pair in assign for x in pair]


def pin_brute_force(m=0):
    for causal in (True, False):
        for (B, H, Hkv, S, D, seed) in ((1, 2, 2, 7, 4, 11), (2, 4, 2, 12, 8, 12),
                                        (1, 3, 1, 16, 5, 13)):
            q, k, v, _ = small(B, H, Hkv, S, D, seed)
            out, lse = oracle.attn_fwd(q, k, v, causal=causal, mutation=m)
            bo, bl = brute.attn_fwd(q.tolist(), k.tolist(), v.tolist(), causal=causal)
            np.testing.assert_allclose(out, np.array(bo), rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse, np.array(bl), rtol=0, atol=1e-12)


def pin_constant_v(m=0):
    q, k, v, _ = small(2, 4, 2, 32, 8, 21)
    v[:] = np.random.default_rng(5).standard_normal((2, 1, 2, 8)).astype(np.float32)
    for causal in (True, False):
        out, _ = oracle.attn_fwd(q, k, v, causal=causal, mutation=m)
        expect = v[:, :, [0, 0, 1, 1], :].astype(np.float64)
        np.testing.assert_allclose(out, expect, rtol=0, atol=1e-12)


def pin_q_zero(m=0):
    B, H, Hkv, S, D = 1, 2, 1, 24, 8
    q, k, v, _ = small(B, H, Hkv, S, D, 22)
    q[:] = 0.0
    vv = v.astype(np.float64)
    for causal in (True, False):
        out, lse = oracle.attn_fwd(q, k, v, causal=causal, mutation=m)
        for i in range(S):
            n = i + 1 if causal else S
            mean = vv[0, :n, 0, :].mean(axis=0)
            for h in range(H):
                np.testing.assert_allclose(out[0, i, h], mean, rtol=0, atol=1e-12)
                assert abs(lse[0, h, i] - math.log(n)) < 1e-12


def pin_row0(m=0):
    q, k, v, _ = small(1, 2, 2, 16, 8, 23)
    out, lse = oracle.attn_fwd(q, k, v, causal=True, mutation=m)
    for h in range(2):
        np.testing.assert_allclose(out[0, 0, h], v[0, 0, h].astype(np.float64), atol=1e-12)
        s00 = float(np.dot(q[0, 0, h].astype(np.float64), k[0, 0, h].astype(np.float64)))
        assert abs(lse[0, h, 0] - s00 / math.sqrt(8)) < 1e-12


def pin_ring_invariance(m=0):
    B, H, Hkv, S, D = 2, 4, 2, 64, 16
    q, k, v, _ = small(B, H, Hkv, S, D, 31)
    for causal in (True, False):
        ref_o, ref_l = oracle.attn_fwd(q, k, v, causal=causal, mutation=m)
        for cp in (1, 2, 4, 8, 16):
            layouts = (oracle.ZIGZAG, oracle.CONTIGUOUS) if S % (2 * cp) == 0 \
                else (oracle.CONTIGUOUS,)
            for layout in layouts:
                for order in (0, 1, 2):
                    o, l = oracle.ring_fwd(q, k, v, cp, layout, causal=causal,
                                           merge_order=order, mutation=m)
                    np.testing.assert_allclose(o, ref_o, rtol=0, atol=1e-12)
                    np.testing.assert_allclose(l, ref_l, rtol=0, atol=1e-12)


def pin_step_partials_merge(m=0):
    B, H, Hkv, S, D = 1, 2, 1, 48, 8
    q, k, v, _ = small(B, H, Hkv, S, D, 32)
    ref_o, ref_l = oracle.attn_fwd(q, k, v, causal=True, mutation=m)
    for layout in (oracle.ZIGZAG, oracle.CONTIGUOUS):
        cp = 4
        acc_o, acc_l = oracle.ring_step(q, k, v, cp, layout, 0, mutation=m)
        for t in range(1, cp):
            po, pl = oracle.ring_step(q, k, v, cp, layout, t, mutation=m)
            acc_o, acc_l = oracle.lse_merge(acc_o, acc_l, po, pl, mutation=m)
        np.testing.assert_allclose(acc_o, ref_o, rtol=0, atol=1e-12)
        np.testing.assert_allclose(acc_l, ref_l, rtol=0, atol=1e-12)


def pin_finite_differences(m=0):
    B, H, Hkv, S, D = 1, 2, 1, 5, 3
    q, k, v, do = small(B, H, Hkv, S, D, 41, dout=True)
    for causal in (True, False):
        dq, dk, dv = oracle.attn_bwd(q, k, v, do, causal=causal, mutation=m)
        ql, kl, vl, dol = (x.astype(np.float64).tolist() for x in (q, k, v, do))
        for name, got in (("q", dq), ("k", dk), ("v", dv)):
            fd = np.array(brute.finite_diff_grad(name, ql, kl, vl, dol, causal=causal))
            np.testing.assert_allclose(got, fd, rtol=0, atol=2e-8)


def pin_sum_rules(m=0):
    B, H, Hkv, S, D = 2, 4, 2, 40, 8
    q, k, v, do = small(B, H, Hkv, S, D, 42, dout=True)
    for causal in (True, False):
        dq, dk, dv = oracle.attn_bwd(q, k, v, do, causal=causal, mutation=m)
        d64 = do.astype(np.float64)
        for g in range(Hkv):
            heads = [h for h in range(H) if h * Hkv // H == g]
            np.testing.assert_allclose(dv[:, :, g].sum(axis=1),
                                       d64[:, :, heads].sum(axis=(1, 2)), atol=1e-10)
            np.testing.assert_allclose(dk[:, :, g].sum(axis=1), 0.0, atol=1e-10)


def pin_key_rows_given_forward(m=0):
    # dK / dV on listed key rows for a dense dO, from the definition's O and
    # LSE: central finite differences of the brute force (two query heads on
    # one kv head, so the sum over the group is exercised) and the sum rules
    # over every key row of a longer problem.
    B, H, Hkv, S, D = 1, 2, 1, 5, 3
    q, k, v, do = small(B, H, Hkv, S, D, 43, dout=True)
    krows = np.array([[0, 0, j] for j in range(S)])
    for causal in (True, False):
        out, lse = oracle.attn_fwd(q, k, v, causal=causal, mutation=m)
        dk, dv = oracle.attn_bwd_dkdv_rows(q, k, v, do, out, lse, krows, causal=causal,
                                           mutation=m)
        ql, kl, vl, dol = (x.astype(np.float64).tolist() for x in (q, k, v, do))
        for name, got in (("k", dk), ("v", dv)):
            fd = np.array(brute.finite_diff_grad(name, ql, kl, vl, dol, causal=causal))
            np.testing.assert_allclose(got, fd[0, :, 0], rtol=0, atol=2e-8)
    B, H, Hkv, S, D = 2, 4, 2, 40, 8
    q, k, v, do = small(B, H, Hkv, S, D, 44, dout=True)
    krows = np.array([[b, g, j] for b in range(B) for g in range(Hkv) for j in range(S)])
    for causal in (True, False):
        out, lse = oracle.attn_fwd(q, k, v, causal=causal, mutation=m)
        dk, dv = oracle.attn_bwd_dkdv_rows(q, k, v, do, out, lse, krows, causal=causal,
                                           mutation=m)
        dk = dk.reshape(B, Hkv, S, D)
        dv = dv.reshape(B, Hkv, S, D)
        d64 = do.astype(np.float64)
        for g in range(Hkv):
            heads = [h for h in range(H) if h * Hkv // H == g]
            np.testing.assert_allclose(dv[:, g].sum(axis=1), d64[:, :, heads].sum(axis=(1, 2)),
                                       atol=1e-10)
            np.testing.assert_allclose(dk[:, g].sum(axis=1), 0.0, atol=1e-10)


def pin_tile_counts(m=0):
    for cp in (1, 2, 4, 8):
        for n in (1, 2, 3):
            T = 4
            c = n * T
            # zigzag, causal: 2n^2 + n tiles at t = 0, 2n^2 after; pairs 2c^2 + c, 2c^2.
            S = 2 * cp * c
            tiles, pairs = oracle.tile_counts(S, cp, oracle.ZIGZAG, True, T, pairs=True,
                                              mutation=m)
            for r in range(cp):
                for t in range(cp):
                    assert tiles[r, t] == (2 * n * n + n if t == 0 else 2 * n * n)
                    assert pairs[r, t] == (2 * c * c + c if t == 0 else 2 * c * c)
            assert int(pairs.sum()) == S * (S + 1) // 2
            # contiguous, causal: L(L+1)/2 at t = 0; L^2 when the source is earlier
            # (t <= r, ring receiving from r - 1), else nothing.
            Lc = 2 * c
            mm = Lc // T
            S = cp * Lc
            tiles, pairs = oracle.tile_counts(S, cp, oracle.CONTIGUOUS, True, T, pairs=True,
                                              mutation=m)
            for r in range(cp):
                for t in range(cp):
                    if t == 0:
                        et, ep = mm * (mm + 1) // 2, Lc * (Lc + 1) // 2
                    elif t <= r:
                        et, ep = mm * mm, Lc * Lc
                    else:
                        et, ep = 0, 0
                    assert tiles[r, t] == et and pairs[r, t] == ep, (cp, n, r, t)
            assert int(pairs.sum()) == S * (S + 1) // 2
            # non-causal: every tile, every pair.
            tiles, pairs = oracle.tile_counts(S, cp, oracle.CONTIGUOUS, False, T, pairs=True,
                                              mutation=m)
            assert (tiles == mm * mm).all() and (pairs == Lc * Lc).all()


# Document offsets used by the pins: a one-token document, documents that
# straddle zigzag chunk borders, and one whose end is the sequence end.
DOCS_S11 = [0, 3, 4, 9, 11]
DOCS_S32 = [0, 5, 6, 13, 24, 32]


def pin_docs_brute_force(m=0):
    for causal in (True, False):
        for (B, H, Hkv, S, D, seed, cu) in ((1, 2, 1, 11, 4, 61, DOCS_S11),
                                            (2, 4, 2, 11, 5, 62, [0, 1, 2, 11]),
                                            (1, 2, 2, 16, 3, 63, [0, 8, 16])):
            q, k, v, _ = small(B, H, Hkv, S, D, seed)
            out, lse = oracle.attn_fwd_docs(q, k, v, cu, causal=causal, mutation=m)
            bo, bl = brute.attn_fwd(q.tolist(), k.tolist(), v.tolist(), causal=causal, docs=cu)
            np.testing.assert_allclose(out, np.array(bo), rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse, np.array(bl), rtol=0, atol=1e-12)


def pin_docs_finite_differences(m=0):
    B, H, Hkv, S, D = 1, 2, 1, 6, 3
    q, k, v, do = small(B, H, Hkv, S, D, 64, dout=True)
    cu = [0, 2, 3, 6]
    for causal in (True, False):
        dq, dk, dv = oracle.attn_bwd_docs(q, k, v, do, cu, causal=causal, mutation=m)
        ql, kl, vl, dol = (x.astype(np.float64).tolist() for x in (q, k, v, do))
        for name, got in (("q", dq), ("k", dk), ("v", dv)):
            fd = np.array(brute.finite_diff_grad(name, ql, kl, vl, dol, causal=causal, docs=cu))
            np.testing.assert_allclose(got, fd, rtol=0, atol=2e-8)


def pin_docs_one_token_each(m=0):
    # Every token its own document: the softmax has one term, so O_i = V_i of
    # the query head's group and LSE_i = scale * q_i . k_i; dQ = dK = 0, dV_i
    # sums dO_i over the group's heads.
    B, H, Hkv, S, D = 2, 4, 2, 12, 8
    q, k, v, do = small(B, H, Hkv, S, D, 65, dout=True)
    cu = list(range(S + 1))
    scale = oracle.default_scale(D)
    grp = [h * Hkv // H for h in range(H)]
    for causal in (True, False):
        out, lse = oracle.attn_fwd_docs(q, k, v, cu, causal=causal, mutation=m)
        np.testing.assert_allclose(out, v[:, :, grp, :].astype(np.float64), rtol=0, atol=1e-12)
        expect = scale * np.einsum("bshd,bshd->bhs", q.astype(np.float64),
                                   k[:, :, grp, :].astype(np.float64))
        np.testing.assert_allclose(lse, expect, rtol=0, atol=1e-12)
        dq, dk, dv = oracle.attn_bwd_docs(q, k, v, do, cu, causal=causal, mutation=m)
        np.testing.assert_allclose(dq, 0.0, atol=1e-12)
        np.testing.assert_allclose(dk, 0.0, atol=1e-12)
        d64 = do.astype(np.float64)
        for g in range(Hkv):
            heads = [h for h in range(H) if grp[h] == g]
            np.testing.assert_allclose(dv[:, :, g], d64[:, :, heads].sum(axis=2), atol=1e-12)


def pin_docs_packed_equals_separate(m=0):
    # Packing documents into one sequence changes nothing for any of them;
    # with the last document taken as padding (large values, dO = 0 there),
    # the real tokens' results equal those of the unpadded sequence.
    B, H, Hkv, S, D = 1, 4, 2, 32, 8
    q, k, v, do = small(B, H, Hkv, S, D, 66, dout=True)
    cu = DOCS_S32
    pad = slice(cu[-2], cu[-1])
    for x in (q, k, v):
        x[:, pad] *= 40.0
    do[:, pad] = 0.0
    for causal in (True, False):
        out, lse = oracle.attn_fwd_docs(q, k, v, cu, causal=causal, mutation=m)
        dq, dk, dv = oracle.attn_bwd_docs(q, k, v, do, cu, causal=causal, mutation=m)
        for a, b in zip(cu[:-1], cu[1:]):
            sl = slice(a, b)
            so, sl_ = oracle.attn_fwd(q[:, sl], k[:, sl], v[:, sl], causal=causal, mutation=m)
            np.testing.assert_allclose(out[:, sl], so, rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse[:, :, sl], sl_, rtol=0, atol=1e-12)
            sq, sk, sv = oracle.attn_bwd(q[:, sl], k[:, sl], v[:, sl], do[:, sl],
                                         causal=causal, mutation=m)
            np.testing.assert_allclose(dq[:, sl], sq, rtol=0, atol=1e-11)
            np.testing.assert_allclose(dk[:, sl], sk, rtol=0, atol=1e-11)
            np.testing.assert_allclose(dv[:, sl], sv, rtol=0, atol=1e-11)
        # The padding document receives no gradient when its dO is zero.
        assert (dq[:, pad] == 0).all() and (dk[:, pad] == 0).all() and (dv[:, pad] == 0).all()


def pin_docs_single_and_ring(m=0):
    # One document is the plain mask; the ring under documents is independent
    # of cp, layout and merge order and equals the definition.
    B, H, Hkv, S, D = 1, 2, 1, 32, 8
    q, k, v, _ = small(B, H, Hkv, S, D, 67)
    for causal in (True, False):
        po, pl = oracle.attn_fwd(q, k, v, causal=causal, mutation=m)
        do_, dl = oracle.attn_fwd_docs(q, k, v, [0, S], causal=causal, mutation=m)
        np.testing.assert_array_equal(do_, po)
        np.testing.assert_array_equal(dl, pl)
        ref_o, ref_l = oracle.attn_fwd_docs(q, k, v, DOCS_S32, causal=causal, mutation=m)
        for cp in (1, 2, 4):
            for layout in (oracle.CONTIGUOUS, oracle.ZIGZAG):
                for order in (0, 1, 2):
                    ro, rl = oracle.ring_fwd_docs(q, k, v, cp, layout, DOCS_S32, causal=causal,
                                                  merge_order=order, mutation=m)
                    np.testing.assert_allclose(ro, ref_o, rtol=0, atol=1e-12)
                    np.testing.assert_allclose(rl, ref_l, rtol=0, atol=1e-12)


def pin_docs_tile_counts(m=0):
    T = 4
    for cp in (1, 2, 4):
        for layout in (oracle.CONTIGUOUS, oracle.ZIGZAG):
            S = 64
            for causal in (True, False):
                # One document is the plain census.
                t1, p1 = oracle.tile_counts_docs(S, cp, layout, causal, [0, S], T, pairs=True,
                                                 mutation=m)
                t0, p0 = oracle.tile_counts(S, cp, layout, causal, T, pairs=True, mutation=m)
                np.testing.assert_array_equal(t1, t0)
                np.testing.assert_array_equal(p1, p0)
                # Pairs per rank: each query sees its document's earlier tokens
                # (causal) or the whole document.
                cu = [0, 3, 11, 12, 20, 45, S]
                tiles, pairs = oracle.tile_counts_docs(S, cp, layout, causal, cu, T, pairs=True,
                                                       mutation=m)
                nat = oracle.shard_order(S, cp, layout, mutation=m)
                start = {p: a for a, b in zip(cu[:-1], cu[1:]) for p in range(a, b)}
                end = {p: b for a, b in zip(cu[:-1], cu[1:]) for p in range(a, b)}
                L = S // cp
                for r in range(cp):
                    mine = nat[r * L:(r + 1) * L]
                    want = sum((i - start[i] + 1) if causal else (end[i] - start[i])
                               for i in mine.tolist())
                    assert int(pairs[r].sum()) == want, (cp, layout, causal, r)
                assert (tiles <= t0).all()
                assert ((pairs == 0) == (tiles == 0)).all()


def _shard(x, order):
    return np.ascontiguousarray(x[:, order])


def pin_allgather(m=0):
    B, H, Hkv, S, D = 1, 2, 1, 32, 4
    q, k, v, do = small(B, H, Hkv, S, D, 68, dout=True)
    for causal in (True, False):
        for cu in (None, DOCS_S32):
            cuo = cu if cu is not None else [0, S]
            ro, rl = oracle.attn_fwd_docs(q, k, v, cuo, causal=causal, mutation=m)
            rq, rk, rv = oracle.attn_bwd_docs(q, k, v, do, cuo, causal=causal, mutation=m)
            for cp in (1, 2, 4):
                for layout in (oracle.CONTIGUOUS, oracle.ZIGZAG):
                    order = oracle.shard_order(S, cp, layout, mutation=m)
                    qs, ks, vs, ds = (_shard(x, order) for x in (q, k, v, do))
                    o, l = oracle.allgather_fwd(qs, ks, vs, cp, layout, causal, cu_seqlens=cu,
                                                mutation=m)
                    np.testing.assert_allclose(o, ro[:, order], rtol=0, atol=1e-12)
                    np.testing.assert_allclose(l, rl[:, :, order], rtol=0, atol=1e-12)
                    gq, gk, gv = oracle.allgather_bwd(qs, ks, vs, ds, cp, layout, causal,
                                                      cu_seqlens=cu, mutation=m)
                    np.testing.assert_allclose(gq, rq[:, order], rtol=0, atol=1e-11)
                    np.testing.assert_allclose(gk, rk[:, order], rtol=0, atol=1e-11)
                    np.testing.assert_allclose(gv, rv[:, order], rtol=0, atol=1e-11)


def pin_ulysses_a2a(m=0):
    B, S, D = 2, 16, 3
    rng = np.random.default_rng(69)
    for H, Hkv, cp in ((8, 2, 4), (8, 4, 2), (8, 8, 8), (4, 1, 1), (8, 2, 8)):
        for layout in (oracle.CONTIGUOUS, oracle.ZIGZAG):
            order = oracle.shard_order(S, cp, layout, mutation=m)
            for kv in (False, True):
                X = Hkv if kv else H
                x = rng.standard_normal((B, S, X, D)).astype(np.float32)
                out = oracle.ulysses_a2a(_shard(x, order), H, Hkv, cp, layout, kv, mutation=m)
                for r in range(cp):
                    # rank r's query heads are the r-th of cp equal slices; its
                    # kv heads are those these query heads read
                    qh = list(range(r * H // cp, (r + 1) * H // cp))
                    heads = sorted({h * Hkv // H for h in qh}) if kv else qh
                    np.testing.assert_array_equal(out[r], x[:, :, heads])


def pin_ulysses(m=0):
    B, H, Hkv, S, D = 1, 8, 2, 32, 4
    q, k, v, do = small(B, H, Hkv, S, D, 70, dout=True)
    for causal in (True, False):
        for cu in (None, DOCS_S32):
            cuo = cu if cu is not None else [0, S]
            ro, rl = oracle.attn_fwd_docs(q, k, v, cuo, causal=causal, mutation=m)
            rq, rk, rv = oracle.attn_bwd_docs(q, k, v, do, cuo, causal=causal, mutation=m)
            for cp in (1, 2, 4, 8):
                for layout in (oracle.CONTIGUOUS, oracle.ZIGZAG):
                    order = oracle.shard_order(S, cp, layout, mutation=m)
                    qs, ks, vs, ds = (_shard(x, order) for x in (q, k, v, do))
                    o, l = oracle.ulysses_fwd(qs, ks, vs, cp, layout, causal, cu_seqlens=cu,
                                              mutation=m)
                    np.testing.assert_allclose(o, ro[:, order], rtol=0, atol=1e-12)
                    np.testing.assert_allclose(l, rl[:, :, order], rtol=0, atol=1e-12)
                    gq, gk, gv = oracle.ulysses_bwd(qs, ks, vs, ds, cp, layout, causal,
                                                    cu_seqlens=cu, mutation=m)
                    np.testing.assert_allclose(gq, rq[:, order], rtol=0, atol=1e-11)
                    np.testing.assert_allclose(gk, rk[:, order], rtol=0, atol=1e-11)
                    np.testing.assert_allclose(gv, rv[:, order], rtol=0, atol=1e-11)


def _level_tokens(S, n_ranks, layout):
    """Natural tokens of each rank, in shard order, for one level of ranks:
    zigzag pairs chunk r with chunk 2n-1-r (the printed assignment's rule,
    restated in the brute-force module), contiguous gives chunk r."""
    if layout == oracle.ZIGZAG:
        chunks = brute.zigzag_assignment(n_ranks)
        c = S // (2 * n_ranks)
    else:
        chunks = [[r] for r in range(n_ranks)]
        c = S // n_ranks
    return [[ch * c + o for ch in rank for o in range(c)] for rank in chunks]


HIER_SIZES = [(2, 2), (2, 4), (4, 2)]


def pin_hier_a2a(m=0):
    # Hierarchical context parallelism, level sizes [A, P] ("Context
    # Parallelism in MegaDLMs", "Hierarchical Context Parallelism"): member a
    # of group p (global rank p*A + a) holds, after the first-level
    # all-to-all, head slice a of the tokens of level-two shard p in that
    # shard's order.  Expected values from the two levels' token lists.
    B, H, D = 2, 8, 4
    for A, P in HIER_SIZES:
        cp = A * P
        S = 4 * cp
        for layout in (oracle.ZIGZAG, oracle.CONTIGUOUS):
            order = np.concatenate(_level_tokens(S, cp, layout))
            inner = _level_tokens(S, P, layout)
            for Hkv in (2, 4, 8):
                for kv in (False, True):
                    X = Hkv if kv else H
                    x = np.arange(B * S * X * D, dtype=np.float32).reshape(B, S, X, D)
                    try:
                        got = oracle.hier_a2a(x[:, order], H, Hkv, A, P, layout, kv, mutation=m)
                    except ValueError as e:
                        raise AssertionError(f"hier_a2a refused [A={A}, P={P}]: {e}")
                    for a in range(A):
                        q0, nq, g0, ng = oracle.ulysses_heads(a, A, H, Hkv)
                        x0, nx = (g0, ng) if kv else (q0, nq)
                        want = np.concatenate([x[:, inner[p], x0:x0 + nx] for p in range(P)],
                                              axis=1)
                        np.testing.assert_array_equal(got[a], want)


def pin_hier(m=0):
    # Hierarchical (a2a+p2p) attention equals the definition, forward and
    # backward, for every level split, layout and mask.
    B, H, S, D = 1, 8, 32, 8
    for A, P in HIER_SIZES:
        for layout in (oracle.ZIGZAG, oracle.CONTIGUOUS):
            for Hkv, causal, cu in ((2, True, None), (4, False, None), (2, True, [0, 5, 19, 32])):
                q, k, v, do = small(B, H, Hkv, S, D, 70 + A * 10 + P, dout=True)
                cuo = [0, S] if cu is None else cu
                ro, rl = oracle.attn_fwd_docs(q, k, v, cuo, causal=causal, mutation=m)
                rq, rk, rv = oracle.attn_bwd_docs(q, k, v, do, cuo, causal=causal, mutation=m)
                order = oracle.shard_order(S, A * P, layout, mutation=m)
                sh = lambda x: np.ascontiguousarray(x[:, order])  # noqa: E731
                try:
                    go, gl = oracle.hier_fwd(sh(q), sh(k), sh(v), A, P, layout, causal,
                                             cu_seqlens=cu, mutation=m)
                    gq, gk, gv = oracle.hier_bwd(sh(q), sh(k), sh(v), sh(do), A, P, layout,
                                                 causal, cu_seqlens=cu, mutation=m)
                except ValueError as e:
                    raise AssertionError(f"hier refused [A={A}, P={P}]: {e}")
                np.testing.assert_allclose(go, ro[:, order], rtol=0, atol=1e-12)
                np.testing.assert_allclose(gl, rl[:, :, order], rtol=0, atol=1e-12)
                for got, ref in ((gq, rq), (gk, rk), (gv, rv)):
                    np.testing.assert_allclose(got, ref[:, order], rtol=0, atol=1e-11)


PINS = [pin_zigzag_golden, pin_contiguous_golden, pin_coverage, pin_brute_force,
        pin_constant_v, pin_q_zero, pin_row0, pin_ring_invariance, pin_step_partials_merge,
        pin_finite_differences, pin_sum_rules, pin_key_rows_given_forward, pin_tile_counts,
        pin_docs_brute_force, pin_docs_finite_differences, pin_docs_one_token_each,
        pin_docs_packed_equals_separate, pin_docs_single_and_ring, pin_docs_tile_counts,
        pin_allgather, pin_ulysses_a2a, pin_ulysses, pin_hier_a2a, pin_hier]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(0)


# ----------------------------------------------------------------------------
# consistency of the sampled-row entry points with the full ones
# ----------------------------------------------------------------------------

def test_rows_match_full():
    B, H, Hkv, S, D = 2, 4, 2, 40, 8
    q, k, v, do = small(B, H, Hkv, S, D, 51, dout=True)
    out, lse = oracle.attn_fwd(q, k, v)
    rows = np.array([[b, h, i] for b in range(B) for h in range(H) for i in (0, 7, 39)])
    ro, rl = oracle.attn_fwd_rows(q, k, v, rows)
    np.testing.assert_array_equal(ro, out[rows[:, 0], rows[:, 2], rows[:, 1]])
    np.testing.assert_array_equal(rl, lse[rows[:, 0], rows[:, 1], rows[:, 2]])
    dq, dk, dv = oracle.attn_bwd(q, k, v, do)
    rdq = oracle.attn_bwd_dq_rows(q, k, v, do, rows)
    np.testing.assert_allclose(rdq, dq[rows[:, 0], rows[:, 2], rows[:, 1]], atol=1e-12)
    # dK / dV from a dO that is zero outside a few query rows.
    qrows = np.array([3, 17, 38])
    sparse = np.zeros_like(do)
    sparse[:, qrows] = do[:, qrows]
    dq2, dk2, dv2 = oracle.attn_bwd(q, k, v, sparse)
    krows = np.array([[b, g, j] for b in range(B) for g in range(Hkv) for j in (0, 3, 20, 38)])
    sdk, sdv = oracle.attn_bwd_dkdv_rows_sparse(q, k, v, sparse, qrows, krows)
    np.testing.assert_allclose(sdk, dk2[krows[:, 0], krows[:, 2], krows[:, 1]], atol=1e-12)
    np.testing.assert_allclose(sdv, dv2[krows[:, 0], krows[:, 2], krows[:, 1]], atol=1e-12)
    # The same under documents.
    cu = [0, 5, 6, 22, 40]
    out, lse = oracle.attn_fwd_docs(q, k, v, cu)
    ro, rl = oracle.attn_fwd_rows_docs(q, k, v, rows, cu)
    np.testing.assert_array_equal(ro, out[rows[:, 0], rows[:, 2], rows[:, 1]])
    np.testing.assert_array_equal(rl, lse[rows[:, 0], rows[:, 1], rows[:, 2]])
    dq, dk, dv = oracle.attn_bwd_docs(q, k, v, do, cu)
    rdq = oracle.attn_bwd_dq_rows_docs(q, k, v, do, rows, cu)
    np.testing.assert_allclose(rdq, dq[rows[:, 0], rows[:, 2], rows[:, 1]], atol=1e-12)
    dq2, dk2, dv2 = oracle.attn_bwd_docs(q, k, v, sparse, cu)
    sdk, sdv = oracle.attn_bwd_dkdv_rows_sparse_docs(q, k, v, sparse, qrows, krows, cu)
    np.testing.assert_allclose(sdk, dk2[krows[:, 0], krows[:, 2], krows[:, 1]], atol=1e-12)
    np.testing.assert_allclose(sdv, dv2[krows[:, 0], krows[:, 2], krows[:, 1]], atol=1e-12)


def test_empty_partial_is_neutral():
    B, S, H, D = 1, 6, 2, 4
    rng = np.random.default_rng(3)
    o = rng.standard_normal((B, S, H, D))
    l = rng.standard_normal((B, H, S))
    zo = np.zeros_like(o)
    zl = np.full_like(l, -np.inf)
    for a, b in (((o, l), (zo, zl)), ((zo, zl), (o, l))):
        mo, ml = oracle.lse_merge(a[0], a[1], b[0], b[1])
        np.testing.assert_array_equal(mo, o)
        np.testing.assert_array_equal(ml, l)
    mo, ml = oracle.lse_merge(zo, zl, zo, zl)
    assert np.isneginf(ml).all() and (mo == 0).all()


def test_bad_arguments_rejected():
    with pytest.raises(ValueError):
        oracle.shard_order(10, 4, oracle.ZIGZAG)
    q, k, v, _ = small(1, 1, 1, 10, 4, 1)
    with pytest.raises(ValueError):
        oracle.ring_fwd(q, k, v, 4, oracle.ZIGZAG)


# ----------------------------------------------------------------------------
# planted mistakes
# ----------------------------------------------------------------------------

MUTATIONS = {1: "wrong zigzag pairing", 2: "interleaved GQA head map",
             3: "causal diagonal dropped", 4: "softmax scale dropped",
             5: "merge term dropped", 6: "ring turned the other way",
             7: "document border off by one", 8: "all-gather reduce drops a rank",
             9: "Ulysses kv heads of the wrong rank",
             10: "key-row gradients drop a query head of the group",
             11: "hierarchical groups of strided ranks (wrong level)"}


@pytest.mark.parametrize("m", sorted(MUTATIONS), ids=[MUTATIONS[m] for m in sorted(MUTATIONS)])
def test_mutations_are_caught(m):
    failed = []
    for pin in PINS:
        try:
            pin(m)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin caught mutation {m} ({MUTATIONS[m]})"
