"""CPU fp64 oracle for context-parallel zigzag causal attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The product
path (``context_causal_attention_zigzag_gb300``) never imports it.

The arithmetic lives in ``cpattn_oracle.c`` (plain C, double precision) and,
for tiny inputs, in the pure-Python ``brute`` module.  This file only moves
numpy arrays across ctypes.  Sources for each function are given in the C
file; in short:

* attention definition and gradients -- "Context Parallelism for Long-Context
  Training", section "Prove attention equivalence";
* chunk placement (zigzag and contiguous), ring step source and per-step
  partials -- "Sequence Parallelism IV: Megatron Context Parallel and
  Load-Balanced Rings", sections 3-5;
* the all-gather schedule, the a2a (Ulysses) variant and hierarchical
  a2a+p2p context parallelism -- "Context Parallelism in MegaDLMs",
  sections "Key-Value Communication Patterns" and "Hierarchical Context
  Parallelism", and "Sequence Parallelism IV", section 7.

Arrays: q [B,S,H,D], k/v [B,S,Hkv,D] float32 (values exactly representable,
e.g. bf16-rounded), natural token order.  Outputs are float64; LSE is
[B,H,S] natural log.
"""
import ctypes
import os

import numpy as np

from . import build as _build

CONTIGUOUS = 0
ZIGZAG = 1

_libs = {}

_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_i64p = np.ctypeslib.ndpointer(dtype=np.int64, flags="C_CONTIGUOUS")
_u64p = np.ctypeslib.ndpointer(dtype=np.uint64, flags="C_CONTIGUOUS")
_L, _I, _D = ctypes.c_long, ctypes.c_int, ctypes.c_double


def _lib(mutation: int = 0):
    if mutation in _libs:
        return _libs[mutation]
    lib = ctypes.CDLL(_build.build(mutation))
    lib.oracle_set_threads.argtypes = [_I]
    lib.oracle_get_threads.restype = _I
    lib.oracle_shard_order.argtypes = [_L, _I, _I, _i64p]
    lib.oracle_shard_order.restype = _I
    shape = [_L, _I, _I, _L, _I, _I, _D]
    lib.oracle_attn_fwd.argtypes = [_f32p, _f32p, _f32p] + shape + [_f64p, _f64p]
    lib.oracle_attn_fwd_rows.argtypes = [_f32p, _f32p, _f32p] + shape + [_i64p, _L, _f64p, _f64p]
    lib.oracle_lse_merge_arrays.argtypes = [_f64p, _f64p, _f64p, _f64p, _L, _L, _I, _I, _f64p, _f64p]
    ring = [_L, _I, _I, _L, _I, _I, _I, _I, _D]
    lib.oracle_ring_step.argtypes = [_f32p, _f32p, _f32p] + ring + [_I, _f64p, _f64p]
    lib.oracle_ring_step.restype = _I
    lib.oracle_ring_fwd.argtypes = [_f32p, _f32p, _f32p] + ring + [_I, _f64p, _f64p]
    lib.oracle_ring_fwd.restype = _I
    lib.oracle_attn_bwd.argtypes = [_f32p] * 4 + shape + [_f64p] * 3
    lib.oracle_attn_bwd_dq_rows.argtypes = [_f32p] * 4 + shape + [_i64p, _L, _f64p]
    lib.oracle_attn_bwd_dkdv_rows_sparse.argtypes = ([_f32p] * 4 + shape
                                                     + [_i64p, _L, _i64p, _L, _f64p, _f64p])
    lib.oracle_attn_bwd_dkdv_rows.argtypes = ([_f32p] * 4 + shape
                                              + [_f64p, _f64p, _i64p, _L, _f64p, _f64p])
    lib.oracle_tile_counts.argtypes = [_L, _I, _I, _I, _L, _u64p, ctypes.c_void_p]
    lib.oracle_tile_counts.restype = _I
    docs = [_i64p, _L]
    lib.oracle_attn_fwd_docs.argtypes = [_f32p, _f32p, _f32p] + shape + docs + [_f64p, _f64p]
    lib.oracle_ring_fwd_docs.argtypes = ([_f32p, _f32p, _f32p] + ring + docs
                                         + [_I, _f64p, _f64p])
    lib.oracle_ring_fwd_docs.restype = _I
    lib.oracle_attn_bwd_docs.argtypes = [_f32p] * 4 + shape + docs + [_f64p] * 3
    lib.oracle_tile_counts_docs.argtypes = ([_L, _I, _I, _I] + docs
                                            + [_L, _u64p, ctypes.c_void_p])
    lib.oracle_tile_counts_docs.restype = _I
    lib.oracle_attn_fwd_rows_docs.argtypes = ([_f32p, _f32p, _f32p] + shape + docs
                                              + [_i64p, _L, _f64p, _f64p])
    lib.oracle_attn_bwd_dq_rows_docs.argtypes = [_f32p] * 4 + shape + docs + [_i64p, _L, _f64p]
    lib.oracle_attn_bwd_dkdv_rows_sparse_docs.argtypes = ([_f32p] * 4 + shape + docs
                                                          + [_i64p, _L, _i64p, _L, _f64p, _f64p])
    lib.oracle_allgather_fwd.argtypes = ([_f32p, _f32p, _f32p] + ring + docs
                                         + [_f64p, _f64p])
    lib.oracle_allgather_fwd.restype = _I
    lib.oracle_allgather_bwd.argtypes = [_f32p] * 4 + ring + docs + [_f64p] * 3
    lib.oracle_allgather_bwd.restype = _I
    _f32o = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS,WRITEABLE")
    lib.oracle_ulysses_a2a.argtypes = [_f32p, _L, _L, _I, _I, _I, _I, _I, _I, _f32o]
    lib.oracle_ulysses_a2a.restype = _I
    lib.oracle_ulysses_fwd.argtypes = [_f32p, _f32p, _f32p] + ring + docs + [_f64p, _f64p]
    lib.oracle_ulysses_fwd.restype = _I
    lib.oracle_ulysses_bwd.argtypes = [_f32p] * 4 + ring + docs + [_f64p] * 3
    lib.oracle_ulysses_bwd.restype = _I
    lib.oracle_hier_a2a.argtypes = [_f32p, _L, _L, _I, _I, _I, _I, _I, _I, _I, _f32o]
    lib.oracle_hier_a2a.restype = _I
    hier = [_L, _I, _I, _L, _I, _I, _I, _I, _I, _D]
    lib.oracle_hier_fwd.argtypes = [_f32p, _f32p, _f32p] + hier + docs + [_f64p, _f64p]
    lib.oracle_hier_fwd.restype = _I
    lib.oracle_hier_bwd.argtypes = [_f32p] * 4 + hier + docs + [_f64p] * 3
    lib.oracle_hier_bwd.restype = _I
    _libs[mutation] = lib
    return lib


def set_threads(n: int, mutation: int = 0) -> None:
    _lib(mutation).oracle_set_threads(int(n))


def get_threads(mutation: int = 0) -> int:
    return int(_lib(mutation).oracle_get_threads())


def _f32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def _shape(q, k):
    B, S, H, D = q.shape
    Hkv = k.shape[2]
    return B, S, H, Hkv, D


def default_scale(D: int) -> float:
    return 1.0 / float(np.sqrt(D))


def shard_order(S: int, cp: int, layout: int, mutation: int = 0) -> np.ndarray:
    """nat[p] = natural position of sharded position p."""
    out = np.empty(S, dtype=np.int64)
    if _lib(mutation).oracle_shard_order(S, cp, layout, out) != 0:
        raise ValueError(f"S={S} does not split into chunks for cp={cp} layout={layout}")
    return out


def attn_fwd(q, k, v, causal=True, scale=None, mutation: int = 0):
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, S, H, Hkv, D = _shape(q, k)
    scale = default_scale(D) if scale is None else scale
    out = np.empty((B, S, H, D), np.float64)
    lse = np.empty((B, H, S), np.float64)
    _lib(mutation).oracle_attn_fwd(q, k, v, B, H, Hkv, S, D, int(causal), scale, out, lse)
    return out, lse


def attn_fwd_rows(q, k, v, rows, causal=True, scale=None, mutation: int = 0):
    """rows: int array [n, 3] of natural (b, h, i).  Returns out [n, D], lse [n]."""
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, S, H, Hkv, D = _shape(q, k)
    scale = default_scale(D) if scale is None else scale
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    n = rows.shape[0]
    out = np.empty((n, D), np.float64)
    lse = np.empty((n,), np.float64)
    _lib(mutation).oracle_attn_fwd_rows(q, k, v, B, H, Hkv, S, D, int(causal), scale, rows, n,
                                        out, lse)
    return out, lse


def lse_merge(o_a, l_a, o_b, l_b, mutation: int = 0):
    """Exact merge of two normalised partials; O [B,S,H,D], LSE [B,H,S]."""
    o_a, o_b = (np.ascontiguousarray(x, dtype=np.float64) for x in (o_a, o_b))
    l_a, l_b = (np.ascontiguousarray(x, dtype=np.float64) for x in (l_a, l_b))
    B, S, H, D = o_a.shape
    o = np.empty_like(o_a)
    lo = np.empty_like(l_a)
    _lib(mutation).oracle_lse_merge_arrays(o_a, l_a, o_b, l_b, B, S, H, D, o, lo)
    return o, lo


def ring_step(q, k, v, cp, layout, t, causal=True, scale=None, mutation: int = 0):
    """Partial (O_rt, L_rt) of ring step t for every rank, natural order."""
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, S, H, Hkv, D = _shape(q, k)
    scale = default_scale(D) if scale is None else scale
    o = np.empty((B, S, H, D), np.float64)
    l = np.empty((B, H, S), np.float64)
    rc = _lib(mutation).oracle_ring_step(q, k, v, B, H, Hkv, S, D, cp, layout, int(causal), scale,
                                         t, o, l)
    if rc != 0:
        raise ValueError("bad ring_step arguments")
    return o, l


def ring_fwd(q, k, v, cp, layout, causal=True, scale=None, merge_order=0, mutation: int = 0):
    """Sequential ring with exact LSE merges; natural order out/lse."""
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, S, H, Hkv, D = _shape(q, k)
    scale = default_scale(D) if scale is None else scale
    out = np.empty((B, S, H, D), np.float64)
    lse = np.empty((B, H, S), np.float64)
    rc = _lib(mutation).oracle_ring_fwd(q, k, v, B, H, Hkv, S, D, cp, layout, int(causal), scale,
                                        merge_order, out, lse)
    if rc != 0:
        raise ValueError("bad ring_fwd arguments")
    return out, lse


def attn_bwd(q, k, v, dout, causal=True, scale=None, mutation: int = 0):
    q, k, v, dout = _f32(q), _f32(k), _f32(v), _f32(dout)
    B, S, H, Hkv, D = _shape(q, k)
    scale = default_scale(D) if scale is None else scale
    dq = np.empty((B, S, H, D), np.float64)
    dk = np.empty((B, S, Hkv, D), np.float64)
    dv = np.empty((B, S, Hkv, D), np.float64)
    _lib(mutation).oracle_attn_bwd(q, k, v, dout, B, H, Hkv, S, D, int(causal), scale, dq, dk, dv)
    return dq, dk, dv


def attn_bwd_dq_rows(q, k, v, dout, rows, causal=True, scale=None, mutation: int = 0):
    q, k, v, dout = _f32(q), _f32(k), _f32(v), _f32(dout)
    B, S, H, Hkv, D = _shape(q, k)
    scale = default_scale(D) if scale is None else scale
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    dq = np.empty((rows.shape[0], D), np.float64)
    _lib(mutation).oracle_attn_bwd_dq_rows(q, k, v, dout, B, H, Hkv, S, D, int(causal), scale,
                                           rows, rows.shape[0], dq)
    return dq


def attn_bwd_dkdv_rows_sparse(q, k, v, dout, qrows, krows, causal=True, scale=None,
                              mutation: int = 0):
    """dK/dV rows (b, g, j) for a dout that is zero outside natural rows qrows."""
    q, k, v, dout = _f32(q), _f32(k), _f32(v), _f32(dout)
    B, S, H, Hkv, D = _shape(q, k)
    scale = default_scale(D) if scale is None else scale
    qrows = np.ascontiguousarray(np.asarray(qrows, dtype=np.int64).reshape(-1))
    krows = np.ascontiguousarray(np.asarray(krows, dtype=np.int64).reshape(-1, 3))
    n = krows.shape[0]
    dk = np.empty((n, D), np.float64)
    dv = np.empty((n, D), np.float64)
    _lib(mutation).oracle_attn_bwd_dkdv_rows_sparse(q, k, v, dout, B, H, Hkv, S, D, int(causal),
                                                    scale, qrows, qrows.shape[0], krows, n, dk, dv)
    return dk, dv


def attn_bwd_dkdv_rows(q, k, v, dout, out, lse, krows, causal=True, scale=None,
                       mutation: int = 0):
    """dK/dV rows (b, g, j) for any dout, from the definition's out [B,S,H,D]
    and lse [B,H,S] of every query row (as ``attn_fwd`` returns them)."""
    q, k, v, dout = _f32(q), _f32(k), _f32(v), _f32(dout)
    B, S, H, Hkv, D = _shape(q, k)
    scale = default_scale(D) if scale is None else scale
    out = np.ascontiguousarray(out, dtype=np.float64)
    lse = np.ascontiguousarray(lse, dtype=np.float64)
    if out.shape != (B, S, H, D) or lse.shape != (B, H, S):
        raise ValueError("out / lse do not match the problem's shape")
    krows = np.ascontiguousarray(np.asarray(krows, dtype=np.int64).reshape(-1, 3))
    n = krows.shape[0]
    dk = np.empty((n, D), np.float64)
    dv = np.empty((n, D), np.float64)
    _lib(mutation).oracle_attn_bwd_dkdv_rows(q, k, v, dout, B, H, Hkv, S, D, int(causal), scale,
                                             out, lse, krows, n, dk, dv)
    return dk, dv


def tile_counts(S, cp, layout, causal, T, pairs=False, mutation: int = 0):
    """(tiles[cp, cp], pairs[cp, cp] or None) per (rank r, ring step t)."""
    tiles = np.zeros(cp * cp, np.uint64)
    pr = np.zeros(cp * cp, np.uint64) if pairs else None
    ptr = pr.ctypes.data_as(ctypes.c_void_p) if pairs else None
    rc = _lib(mutation).oracle_tile_counts(S, cp, layout, int(causal), T, tiles, ptr)
    if rc != 0:
        raise ValueError("bad tile_counts arguments")
    return tiles.reshape(cp, cp), (pr.reshape(cp, cp) if pairs else None)


def _cu(cu_seqlens, S):
    """Document offsets as int64; checks cu[0] = 0, cu[-1] = S, increasing."""
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64).reshape(-1))
    if cu.size < 2 or cu[0] != 0 or cu[-1] != S or np.any(np.diff(cu) <= 0):
        raise ValueError(f"cu_seqlens must rise strictly from 0 to S={S}: {cu.tolist()}")
    return cu, cu.size - 1


def attn_fwd_docs(q, k, v, cu_seqlens, causal=True, scale=None, mutation: int = 0):
    """The definition under the document rule: documents [cu[d], cu[d+1])."""
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, S, H, Hkv, D = _shape(q, k)
    cu, nd = _cu(cu_seqlens, S)
    scale = default_scale(D) if scale is None else scale
    out = np.empty((B, S, H, D), np.float64)
    lse = np.empty((B, H, S), np.float64)
    _lib(mutation).oracle_attn_fwd_docs(q, k, v, B, H, Hkv, S, D, int(causal), scale, cu, nd,
                                        out, lse)
    return out, lse


def ring_fwd_docs(q, k, v, cp, layout, cu_seqlens, causal=True, scale=None, merge_order=0,
                  mutation: int = 0):
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, S, H, Hkv, D = _shape(q, k)
    cu, nd = _cu(cu_seqlens, S)
    scale = default_scale(D) if scale is None else scale
    out = np.empty((B, S, H, D), np.float64)
    lse = np.empty((B, H, S), np.float64)
    rc = _lib(mutation).oracle_ring_fwd_docs(q, k, v, B, H, Hkv, S, D, cp, layout, int(causal),
                                             scale, cu, nd, merge_order, out, lse)
    if rc != 0:
        raise ValueError("bad ring_fwd_docs arguments")
    return out, lse


def attn_bwd_docs(q, k, v, dout, cu_seqlens, causal=True, scale=None, mutation: int = 0):
    q, k, v, dout = _f32(q), _f32(k), _f32(v), _f32(dout)
    B, S, H, Hkv, D = _shape(q, k)
    cu, nd = _cu(cu_seqlens, S)
    scale = default_scale(D) if scale is None else scale
    dq = np.empty((B, S, H, D), np.float64)
    dk = np.empty((B, S, Hkv, D), np.float64)
    dv = np.empty((B, S, Hkv, D), np.float64)
    _lib(mutation).oracle_attn_bwd_docs(q, k, v, dout, B, H, Hkv, S, D, int(causal), scale, cu,
                                        nd, dq, dk, dv)
    return dq, dk, dv


def tile_counts_docs(S, cp, layout, causal, cu_seqlens, T, pairs=False, mutation: int = 0):
    """tile_counts under the document rule (every pair of a tile enumerated)."""
    cu, nd = _cu(cu_seqlens, S)
    tiles = np.zeros(cp * cp, np.uint64)
    pr = np.zeros(cp * cp, np.uint64) if pairs else None
    ptr = pr.ctypes.data_as(ctypes.c_void_p) if pairs else None
    rc = _lib(mutation).oracle_tile_counts_docs(S, cp, layout, int(causal), cu, nd, T, tiles, ptr)
    if rc != 0:
        raise ValueError("bad tile_counts_docs arguments")
    return tiles.reshape(cp, cp), (pr.reshape(cp, cp) if pairs else None)


def attn_fwd_rows_docs(q, k, v, rows, cu_seqlens, causal=True, scale=None, mutation: int = 0):
    """attn_fwd_rows under the document rule."""
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, S, H, Hkv, D = _shape(q, k)
    cu, nd = _cu(cu_seqlens, S)
    scale = default_scale(D) if scale is None else scale
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    n = rows.shape[0]
    out = np.empty((n, D), np.float64)
    lse = np.empty((n,), np.float64)
    _lib(mutation).oracle_attn_fwd_rows_docs(q, k, v, B, H, Hkv, S, D, int(causal), scale, cu, nd,
                                             rows, n, out, lse)
    return out, lse


def attn_bwd_dq_rows_docs(q, k, v, dout, rows, cu_seqlens, causal=True, scale=None,
                          mutation: int = 0):
    q, k, v, dout = _f32(q), _f32(k), _f32(v), _f32(dout)
    B, S, H, Hkv, D = _shape(q, k)
    cu, nd = _cu(cu_seqlens, S)
    scale = default_scale(D) if scale is None else scale
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    dq = np.empty((rows.shape[0], D), np.float64)
    _lib(mutation).oracle_attn_bwd_dq_rows_docs(q, k, v, dout, B, H, Hkv, S, D, int(causal),
                                                scale, cu, nd, rows, rows.shape[0], dq)
    return dq


def attn_bwd_dkdv_rows_sparse_docs(q, k, v, dout, qrows, krows, cu_seqlens, causal=True,
                                   scale=None, mutation: int = 0):
    q, k, v, dout = _f32(q), _f32(k), _f32(v), _f32(dout)
    B, S, H, Hkv, D = _shape(q, k)
    cu, nd = _cu(cu_seqlens, S)
    scale = default_scale(D) if scale is None else scale
    qrows = np.ascontiguousarray(np.asarray(qrows, dtype=np.int64).reshape(-1))
    krows = np.ascontiguousarray(np.asarray(krows, dtype=np.int64).reshape(-1, 3))
    n = krows.shape[0]
    dk = np.empty((n, D), np.float64)
    dv = np.empty((n, D), np.float64)
    _lib(mutation).oracle_attn_bwd_dkdv_rows_sparse_docs(q, k, v, dout, B, H, Hkv, S, D,
                                                         int(causal), scale, cu, nd, qrows,
                                                         qrows.shape[0], krows, n, dk, dv)
    return dk, dv


def _cu_or_one(cu_seqlens, S):
    return _cu(cu_seqlens if cu_seqlens is not None else [0, S], S)


def allgather_fwd(q_sh, k_sh, v_sh, cp, layout, causal=True, scale=None, cu_seqlens=None,
                  mutation: int = 0):
    """The all-gather schedule on SHARDED-order inputs: every rank gathers the
    whole K/V, then attends its own queries to it in one pass.  Returns
    (out, lse) in sharded order."""
    q, k, v = _f32(q_sh), _f32(k_sh), _f32(v_sh)
    B, S, H, Hkv, D = _shape(q, k)
    cu, nd = _cu_or_one(cu_seqlens, S)
    scale = default_scale(D) if scale is None else scale
    out = np.empty((B, S, H, D), np.float64)
    lse = np.empty((B, H, S), np.float64)
    rc = _lib(mutation).oracle_allgather_fwd(q, k, v, B, H, Hkv, S, D, cp, layout, int(causal),
                                             scale, cu, nd, out, lse)
    if rc != 0:
        raise ValueError("bad allgather_fwd arguments")
    return out, lse


def allgather_bwd(q_sh, k_sh, v_sh, do_sh, cp, layout, causal=True, scale=None, cu_seqlens=None,
                  mutation: int = 0):
    """Backward of the all-gather schedule, sharded order in and out: per-rank
    dK/dV contributions summed over ranks, each rank keeping its shard."""
    q, k, v, do = _f32(q_sh), _f32(k_sh), _f32(v_sh), _f32(do_sh)
    B, S, H, Hkv, D = _shape(q, k)
    cu, nd = _cu_or_one(cu_seqlens, S)
    scale = default_scale(D) if scale is None else scale
    dq = np.empty((B, S, H, D), np.float64)
    dk = np.empty((B, S, Hkv, D), np.float64)
    dv = np.empty((B, S, Hkv, D), np.float64)
    rc = _lib(mutation).oracle_allgather_bwd(q, k, v, do, B, H, Hkv, S, D, cp, layout,
                                             int(causal), scale, cu, nd, dq, dk, dv)
    if rc != 0:
        raise ValueError("bad allgather_bwd arguments")
    return dq, dk, dv


def ulysses_heads(r, cp, H, Hkv):
    """(first query head, count, first kv head, count) of rank r after the
    sequence-to-head all-to-all (as the C oracle assigns them)."""
    hc, grp = H // cp, H // Hkv
    return r * hc, hc, (r * hc) // grp, (hc // grp if hc >= grp else 1)


def ulysses_a2a(x_sh, H, Hkv, cp, layout, kv=False, mutation: int = 0):
    """Sequence-to-head all-to-all of a sharded [B,S,X,D] tensor: returns
    [cp, B, S, nx, D], rank r's head slice of every token in natural order."""
    x = _f32(x_sh)
    B, S, X, D = x.shape
    nx = ulysses_heads(0, cp, H, Hkv)[3 if kv else 1]
    out = np.empty((cp, B, S, nx, D), np.float32)
    rc = _lib(mutation).oracle_ulysses_a2a(x, B, S, H, Hkv, D, cp, layout, int(kv), out)
    if rc != 0:
        raise ValueError("bad ulysses_a2a arguments")
    return out


def ulysses_fwd(q_sh, k_sh, v_sh, cp, layout, causal=True, scale=None, cu_seqlens=None,
                mutation: int = 0):
    """Ulysses attention on sharded-order inputs: all-to-all to head owners,
    full attention per head slice, all-to-all back.  Sharded (out, lse)."""
    q, k, v = _f32(q_sh), _f32(k_sh), _f32(v_sh)
    B, S, H, Hkv, D = _shape(q, k)
    cu, nd = _cu_or_one(cu_seqlens, S)
    scale = default_scale(D) if scale is None else scale
    out = np.empty((B, S, H, D), np.float64)
    lse = np.empty((B, H, S), np.float64)
    rc = _lib(mutation).oracle_ulysses_fwd(q, k, v, B, H, Hkv, S, D, cp, layout, int(causal),
                                           scale, cu, nd, out, lse)
    if rc != 0:
        raise ValueError("bad ulysses_fwd arguments")
    return out, lse


def ulysses_bwd(q_sh, k_sh, v_sh, do_sh, cp, layout, causal=True, scale=None, cu_seqlens=None,
                mutation: int = 0):
    q, k, v, do = _f32(q_sh), _f32(k_sh), _f32(v_sh), _f32(do_sh)
    B, S, H, Hkv, D = _shape(q, k)
    cu, nd = _cu_or_one(cu_seqlens, S)
    scale = default_scale(D) if scale is None else scale
    dq = np.empty((B, S, H, D), np.float64)
    dk = np.empty((B, S, Hkv, D), np.float64)
    dv = np.empty((B, S, Hkv, D), np.float64)
    rc = _lib(mutation).oracle_ulysses_bwd(q, k, v, do, B, H, Hkv, S, D, cp, layout, int(causal),
                                           scale, cu, nd, dq, dk, dv)
    if rc != 0:
        raise ValueError("bad ulysses_bwd arguments")
    return dq, dk, dv


def hier_a2a(x_sh, H, Hkv, A, P, layout, kv=False, mutation: int = 0):
    """First-level all-to-all of hierarchical context parallelism (level sizes
    [A, P], cp = A*P) on a [B,S,X,D] tensor sharded over cp ranks: returns
    [A, B, S, nx, D]; block a holds member a's head slice, rows
    [p*S/P, (p+1)*S/P) being what member a of group p holds, in the order of
    level-two shard p."""
    x = _f32(x_sh)
    B, S, X, D = x.shape
    nx = ulysses_heads(0, A, H, Hkv)[3 if kv else 1]
    out = np.empty((A, B, S, nx, D), np.float32)
    rc = _lib(mutation).oracle_hier_a2a(x, B, S, H, Hkv, D, A, P, layout, int(kv), out)
    if rc != 0:
        raise ValueError("bad hier_a2a arguments")
    return out


def hier_fwd(q_sh, k_sh, v_sh, A, P, layout, causal=True, scale=None, cu_seqlens=None,
             mutation: int = 0):
    """Hierarchical (a2a+p2p) attention on inputs sharded over cp = A*P
    ranks: all-to-all inside groups of A, ring over the P groups on each
    head slice, all-to-all back.  Sharded (out, lse)."""
    q, k, v = _f32(q_sh), _f32(k_sh), _f32(v_sh)
    B, S, H, Hkv, D = _shape(q, k)
    cu, nd = _cu_or_one(cu_seqlens, S)
    scale = default_scale(D) if scale is None else scale
    out = np.empty((B, S, H, D), np.float64)
    lse = np.empty((B, H, S), np.float64)
    rc = _lib(mutation).oracle_hier_fwd(q, k, v, B, H, Hkv, S, D, A, P, layout, int(causal),
                                        scale, cu, nd, out, lse)
    if rc != 0:
        raise ValueError("bad hier_fwd arguments")
    return out, lse


def hier_bwd(q_sh, k_sh, v_sh, do_sh, A, P, layout, causal=True, scale=None, cu_seqlens=None,
             mutation: int = 0):
    q, k, v, do = _f32(q_sh), _f32(k_sh), _f32(v_sh), _f32(do_sh)
    B, S, H, Hkv, D = _shape(q, k)
    cu, nd = _cu_or_one(cu_seqlens, S)
    scale = default_scale(D) if scale is None else scale
    dq = np.empty((B, S, H, D), np.float64)
    dk = np.empty((B, S, Hkv, D), np.float64)
    dv = np.empty((B, S, Hkv, D), np.float64)
    rc = _lib(mutation).oracle_hier_bwd(q, k, v, do, B, H, Hkv, S, D, A, P, layout, int(causal),
                                        scale, cu, nd, dq, dk, dv)
    if rc != 0:
        raise ValueError("bad hier_bwd arguments")
    return dq, dk, dv
