"""Pure-Python brute force for tiny inputs (S <= 16): test infrastructure only.

Independent of ``cpattn_oracle.c``: nested Python lists and ``math`` only.
It evaluates softmax attention straight from its definition (every score,
one ``math.exp`` each, normalised by the plain sum -- no max shift, no log
domain) and gives gradients by central finite differences of that forward,
so that it shares neither code nor formulas with the C oracle's backward.
The definition is the unsharded reference of "Context Parallelism for
Long-Context Training", section "Prove attention equivalence".
"""
import math


def _doc_ids(S, docs):
    """Document number of every position; docs lists the offsets
    [0, ..., S] of packed documents, None for one document."""
    if docs is None:
        return [0] * S
    ids = []
    for d in range(len(docs) - 1):
        ids.extend([d] * (docs[d + 1] - docs[d]))
    assert len(ids) == S
    return ids


def attn_fwd(q, k, v, causal=True, scale=None, docs=None):
    """q[b][s][h][d], k/v[b][s][g][d] nested lists.  Returns (out, lse)
    with out[b][s][h][d] and lse[b][h][s] (natural log).  With ``docs`` a
    token sees only the tokens of its own packed document."""
    B, S, H, D = len(q), len(q[0]), len(q[0][0]), len(q[0][0][0])
    Hkv = len(k[0][0])
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    out = [[[[0.0] * D for _ in range(H)] for _ in range(S)] for _ in range(B)]
    lse = [[[0.0] * S for _ in range(H)] for _ in range(B)]
    doc = _doc_ids(S, docs)
    for b in range(B):
        for h in range(H):
            g = (h * Hkv) // H
            for i in range(S):
                weights = []
                for j in range(S):
                    if causal and j > i:
                        continue
                    if doc[j] != doc[i]:
                        continue
                    s = scale * sum(q[b][i][h][d] * k[b][j][g][d] for d in range(D))
                    weights.append((j, math.exp(s)))
                z = sum(w for _, w in weights)
                lse[b][h][i] = math.log(z)
                for d in range(D):
                    out[b][i][h][d] = sum(w * v[b][j][g][d] for j, w in weights) / z
    return out, lse


def loss(q, k, v, dout, causal=True, scale=None, docs=None):
    """L = sum over every element of dout * O: its gradient w.r.t. O is dout."""
    out, _ = attn_fwd(q, k, v, causal, scale, docs)
    B, S, H, D = len(out), len(out[0]), len(out[0][0]), len(out[0][0][0])
    return sum(dout[b][s][h][d] * out[b][s][h][d]
               for b in range(B) for s in range(S) for h in range(H) for d in range(D))


def finite_diff_grad(which, q, k, v, dout, causal=True, scale=None, eps=1e-5, docs=None):
    """Central differences of ``loss`` with respect to one input ('q', 'k', 'v')."""
    import copy
    tensors = {"q": q, "k": k, "v": v}
    base = tensors[which]
    grad = copy.deepcopy(base)
    B, S, X, D = len(base), len(base[0]), len(base[0][0]), len(base[0][0][0])
    for b in range(B):
        for s in range(S):
            for x in range(X):
                for d in range(D):
                    saved = base[b][s][x][d]
                    base[b][s][x][d] = saved + eps
                    lp = loss(tensors["q"], tensors["k"], tensors["v"], dout, causal, scale, docs)
                    base[b][s][x][d] = saved - eps
                    lm = loss(tensors["q"], tensors["k"], tensors["v"], dout, causal, scale, docs)
                    base[b][s][x][d] = saved
                    grad[b][s][x][d] = (lp - lm) / (2 * eps)
    return grad


def zigzag_assignment(cp):
    """Chunks per rank read off the pairing rule: 2*cp chunks, the i-th
    earliest chunk goes with the i-th latest one."""
    early = list(range(cp))
    late = list(range(2 * cp - 1, cp - 1, -1))
    return [[early[r], late[r]] for r in range(cp)]
