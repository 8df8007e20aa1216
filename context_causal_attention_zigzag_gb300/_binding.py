"""ctypes binding of libcpattn (include/cpattn.h): argument marshalling only.

Every step of the path runs in the library's CUDA kernels; this module only
checks tensor dtypes/devices/shapes, allocates outputs with torch (device
memory plumbing) and passes raw pointers plus the current CUDA stream.  If
the library has not been built, every call raises: there is no fallback.
"""
import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libcpattn.so")

OK = 0
ERR_INVALID_ARG = -1
ERR_UNSUPPORTED = -2
ERR_CUDA = -3
ERR_DEVICE_TIMEOUT = -4
ERR_WORKSPACE = -5

CONTIGUOUS = 0
ZIGZAG = 1
F32 = 0
BF16 = 1
GRAD_F32 = 0x10  # OR into the backward's dtype: dq, dk, dv written as float32
ONEPASS = 0x20   # OR into the backward's dtype: one-pass tensor-core backward (dQ by reductions)
PATH_SIMT = 0
PATH_TCGEN05 = 1

# Every entry point include/cpattn.h declares, with its ctypes signature.
_vp, _i, _i64, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
_ip = ctypes.POINTER(ctypes.c_int)
SIGNATURES = {
    "cpattn_zigzag_permute": (_i, [_vp, _vp, _i64, _i64, _i64, _i, _i, _vp]),
    "cpattn_zigzag_unpermute": (_i, [_vp, _vp, _i64, _i64, _i64, _i, _i, _vp]),
    "cpattn_zigzag_permute_pad": (_i, [_vp, _vp, _i64, _i64, _i64, _i64, _i, _i, _vp]),
    "cpattn_zigzag_unpermute_pad": (_i, [_vp, _vp, _i64, _i64, _i64, _i64, _i, _i, _vp]),
    "cpattn_doc_bounds": (_i, [_vp, _i, _i, _vp, _vp]),
    "cpattn_ring_fwd_docs": (_i, [_vp] * 5 + [_i] * 9 + [_f, _vp, _vp, _vp]),
    "cpattn_ring_bwd_docs": (_i, [_vp] * 9 + [_i] * 9 + [_f, _vp, _vp, _sz, _vp]),
    "cpattn_padded_length": (_i64, [_i64, _i, _i]),
    "cpattn_allgather_fwd": (_i, [_vp] * 5 + [_i] * 9 + [_f, _vp, _vp, _vp]),
    "cpattn_allgather_bwd": (_i, [_vp] * 9 + [_i] * 9 + [_f, _vp, _vp, _sz, _vp]),
    "cpattn_ulysses_a2a": (_i, [_vp, _vp] + [_i] * 10 + [_vp]),
    "cpattn_ulysses_lse_a2a": (_i, [_vp, _vp] + [_i] * 6 + [_vp]),
    "cpattn_ulysses_workspace_bytes": (_sz, [_i] * 9),
    "cpattn_ulysses_fwd": (_i, [_vp] * 5 + [_i] * 9 + [_f, _vp, _vp, _sz, _vp]),
    "cpattn_ulysses_bwd": (_i, [_vp] * 9 + [_i] * 9 + [_f, _vp, _vp, _sz, _vp]),
    "cpattn_hier_a2a": (_i, [_vp, _vp] + [_i] * 11 + [_vp]),
    "cpattn_hier_lse_a2a": (_i, [_vp, _vp] + [_i] * 7 + [_vp]),
    "cpattn_hier_workspace_bytes": (_sz, [_i] * 10),
    "cpattn_hier_fwd": (_i, [_vp] * 5 + [_i] * 10 + [_f, _vp, _vp, _sz, _vp]),
    "cpattn_hier_bwd": (_i, [_vp] * 9 + [_i] * 10 + [_f, _vp, _vp, _sz, _vp]),
    "cpattn_attention_host_workspace_bytes": (_sz, [_i] * 9),
    "cpattn_attention_host_parts": (_i, [_i] * 5),
    "cpattn_attention_host_docs_workspace_bytes": (_sz, [_i] * 9),
    "cpattn_attention_host_docs": (_i, [_vp] * 9 + [_i] * 9 + [_f, _vp, _i, _i, _vp, _sz, _vp]),
    "cpattn_attention_host": (_i, [_vp] * 9 + [_i] * 9 + [_f, _i, _vp, _sz, _vp]),
    "cpattn_ring_fwd": (_i, [_vp, _vp, _vp, _vp, _vp] + [_i] * 9 + [_f, _vp]),
    "cpattn_ring_fwd_census": (_i, [_vp, _vp, _vp, _vp, _vp] + [_i] * 9 + [_f, _vp, _vp]),
    "cpattn_ring_fwd_plan": (_i, [_i] * 9 + [_ip, _ip]),
    "cpattn_ring_bwd_plan": (_i, [_i] * 9 + [_ip, _ip]),
    "cpattn_ring_fwd_step": (_i, [_vp, _vp, _vp] + [_i] * 9 + [_f, _i, _vp, _vp, _vp]),
    "cpattn_lse_merge": (_i, [_vp] * 6 + [_i] * 4 + [_vp]),
    "cpattn_ring_bwd_workspace_bytes": (_sz, [_i] * 6),
    "cpattn_ring_bwd": (_i, [_vp] * 9 + [_i] * 9 + [_f, _vp, _sz, _vp]),
    "cpattn_ring_bwd_noalloc": (_i, [_vp] * 9 + [_i] * 9 + [_f, _vp]),
    "cpattn_ring_bwd_census": (_i, [_vp] * 9 + [_i] * 9 + [_f, _vp, _sz, _vp, _vp, _vp]),
    "cpattn_tile_counts": (_i, [_i64, _i, _i, _i, _i64, _vp, _vp]),
    "cpattn_device_status": (_i, [_vp]),
    "cpattn_wait_probe": (_i, [_i64, _vp]),
    "cpattn_status_string": (ctypes.c_char_p, [_i]),
}

_lib = None


class CpattnError(RuntimeError):
    def __init__(self, fn, code):
        self.code = code
        msg = status_string(code) if _lib is not None else str(code)
        super().__init__(f"{fn} failed: {msg} ({code})")


def lib():
    """Loads libcpattn.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    handle = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(handle, name)
        fn.restype = res
        fn.argtypes = args
    _lib = handle
    return handle


def status_string(code: int) -> str:
    return lib().cpattn_status_string(int(code)).decode()


def _check(fn, code):
    if code != OK:
        raise CpattnError(fn, code)


def _stream(t: torch.Tensor = None):
    dev = t.device if t is not None else torch.device("cuda", torch.cuda.current_device())
    return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"unsupported dtype {t.dtype}: bfloat16 or float32")


def _need_cuda(*ts):
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("tensor must be on a CUDA device")
        if not t.is_contiguous():
            raise ValueError("tensor must be contiguous")


def _scale(scale):
    return 0.0 if scale is None else float(scale)


# ---------------------------------------------------------------------------
# permutation
# ---------------------------------------------------------------------------

def _perm(name, x, cp, layout, seq_dim, out):
    _need_cuda(x)
    if seq_dim < 0:
        seq_dim += x.dim()
    outer = 1
    for s in x.shape[:seq_dim]:
        outer *= s
    S = x.shape[seq_dim]
    inner = x.element_size()
    for s in x.shape[seq_dim + 1:]:
        inner *= s
    if out is None:
        out = torch.empty_like(x)
    _need_cuda(out)
    rc = getattr(lib(), name)(_ptr(x), _ptr(out), outer, S, inner, int(cp), int(layout),
                              _stream(x))
    _check(name, rc)
    return out


def zigzag_permute(x, cp, layout=ZIGZAG, seq_dim=1, out=None):
    """Natural -> sharded order along ``seq_dim`` (see cpattn_zigzag_permute)."""
    return _perm("cpattn_zigzag_permute", x, cp, layout, seq_dim, out)


def zigzag_unpermute(x, cp, layout=ZIGZAG, seq_dim=1, out=None):
    """Sharded -> natural order along ``seq_dim``."""
    return _perm("cpattn_zigzag_unpermute", x, cp, layout, seq_dim, out)


def _split(x, seq_dim):
    if seq_dim < 0:
        seq_dim += x.dim()
    outer = 1
    for s in x.shape[:seq_dim]:
        outer *= s
    inner = x.element_size()
    for s in x.shape[seq_dim + 1:]:
        inner *= s
    return seq_dim, outer, inner


def zigzag_permute_pad(x, cp, S, layout=ZIGZAG, seq_dim=1, out=None):
    """Natural [.., S_real, ..] -> sharded [.., S, ..], padding positions
    S_real..S-1 with zeros (cpattn_zigzag_permute_pad)."""
    _need_cuda(x)
    seq_dim, outer, inner = _split(x, seq_dim)
    S_real = x.shape[seq_dim]
    if out is None:
        shape = list(x.shape)
        shape[seq_dim] = S
        out = torch.empty(shape, device=x.device, dtype=x.dtype)
    _need_cuda(out)
    rc = lib().cpattn_zigzag_permute_pad(_ptr(x), _ptr(out), outer, S_real, int(S), inner,
                                         int(cp), int(layout), _stream(x))
    _check("cpattn_zigzag_permute_pad", rc)
    return out


def zigzag_unpermute_pad(x, cp, S_real, layout=ZIGZAG, seq_dim=1, out=None):
    """Sharded [.., S, ..] -> natural [.., S_real, ..], dropping the padding."""
    _need_cuda(x)
    seq_dim, outer, inner = _split(x, seq_dim)
    S = x.shape[seq_dim]
    if out is None:
        shape = list(x.shape)
        shape[seq_dim] = S_real
        out = torch.empty(shape, device=x.device, dtype=x.dtype)
    _need_cuda(out)
    rc = lib().cpattn_zigzag_unpermute_pad(_ptr(x), _ptr(out), outer, int(S_real), S, inner,
                                           int(cp), int(layout), _stream(x))
    _check("cpattn_zigzag_unpermute_pad", rc)
    return out


def padded_length(S, cp, layout=ZIGZAG) -> int:
    """Length the tensor-core kernels take for S tokens (cpattn_padded_length)."""
    n = int(lib().cpattn_padded_length(int(S), int(cp), int(layout)))
    if n < 0:
        raise ValueError(f"bad arguments to padded_length: S={S} cp={cp} layout={layout}")
    return n


# ---------------------------------------------------------------------------
# forward
# ---------------------------------------------------------------------------

def _shape(q, k, v):
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be [B, S, H, D]")
    B, S, H, D = q.shape
    if k.shape != v.shape or k.shape[0] != B or k.shape[1] != S or k.shape[3] != D:
        raise ValueError("k, v must be [B, S, Hkv, D] matching q")
    if q.dtype != k.dtype or q.dtype != v.dtype:
        raise ValueError("q, k, v must share a dtype")
    return B, H, k.shape[2], S, D


def ring_fwd(q, k, v, cp, layout=ZIGZAG, causal=True, scale=None, out=None, lse=None,
             tiles_rt=None):
    """Ring forward on sharded-order tensors; returns (out, lse)."""
    _need_cuda(q, k, v)
    B, H, Hkv, S, D = _shape(q, k, v)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, S), device=q.device, dtype=torch.float32)
    _need_cuda(out, lse)
    args = [_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Hkv, S, D, int(cp),
            int(layout), int(bool(causal)), _dtype_code(q), _scale(scale)]
    if tiles_rt is None:
        rc = lib().cpattn_ring_fwd(*args, _stream(q))
        _check("cpattn_ring_fwd", rc)
    else:
        _need_cuda(tiles_rt)
        rc = lib().cpattn_ring_fwd_census(*args, _ptr(tiles_rt), _stream(q))
        _check("cpattn_ring_fwd_census", rc)
    return out, lse


def ring_fwd_census(q, k, v, cp, layout=ZIGZAG, causal=True, scale=None):
    """Forward plus the kernel's own per-(rank, step) tile counts [cp, cp]."""
    counts = torch.zeros((cp, cp), device=q.device, dtype=torch.int64)
    out, lse = ring_fwd(q, k, v, cp, layout, causal, scale, tiles_rt=counts)
    return out, lse, counts


def ring_fwd_step(q, k, v, cp, step, layout=ZIGZAG, causal=True, scale=None, o_part=None,
                  lse_part=None):
    """Partial (o_part, lse_part) of one ring step for every rank (float32)."""
    _need_cuda(q, k, v)
    B, H, Hkv, S, D = _shape(q, k, v)
    if o_part is None:
        o_part = torch.empty((B, S, H, D), device=q.device, dtype=torch.float32)
    if lse_part is None:
        lse_part = torch.empty((B, H, S), device=q.device, dtype=torch.float32)
    _need_cuda(o_part, lse_part)
    rc = lib().cpattn_ring_fwd_step(_ptr(q), _ptr(k), _ptr(v), B, H, Hkv, S, D, int(cp),
                                    int(layout), int(bool(causal)), _dtype_code(q),
                                    _scale(scale), int(step), _ptr(o_part), _ptr(lse_part),
                                    _stream(q))
    _check("cpattn_ring_fwd_step", rc)
    return o_part, lse_part


def lse_merge(o_a, lse_a, o_b, lse_b, o_out=None, lse_out=None):
    """Exact merge of two partials; o_out/lse_out may alias the inputs."""
    _need_cuda(o_a, lse_a, o_b, lse_b)
    B, S, H, D = o_a.shape
    if o_out is None:
        o_out = torch.empty_like(o_a)
    if lse_out is None:
        lse_out = torch.empty_like(lse_a)
    rc = lib().cpattn_lse_merge(_ptr(o_a), _ptr(lse_a), _ptr(o_b), _ptr(lse_b), _ptr(o_out),
                                _ptr(lse_out), B, S, H, D, _stream(o_a))
    _check("cpattn_lse_merge", rc)
    return o_out, lse_out


def plan(B, H, Hkv, S, D, cp, layout, causal, dtype, backward=False):
    """(path, tile) the library picks for these arguments (host only)."""
    path, tile = ctypes.c_int(-1), ctypes.c_int(-1)
    fn = "cpattn_ring_bwd_plan" if backward else "cpattn_ring_fwd_plan"
    code = dtype if isinstance(dtype, int) else (BF16 if dtype == torch.bfloat16 else F32)
    rc = getattr(lib(), fn)(B, H, Hkv, S, D, int(cp), int(layout), int(bool(causal)), code,
                            ctypes.byref(path), ctypes.byref(tile))
    _check(fn, rc)
    return path.value, tile.value


# ---------------------------------------------------------------------------
# backward
# ---------------------------------------------------------------------------

def ring_bwd_workspace_bytes(B, H, Hkv, S, D, dtype=BF16) -> int:
    return int(lib().cpattn_ring_bwd_workspace_bytes(B, H, Hkv, S, D, int(dtype)))


def _grad_args(q, k, v, dq, dk, dv, grad_dtype, onepass=False):
    code = _dtype_code(q) | (ONEPASS if onepass else 0)
    gdt = q.dtype if grad_dtype is None else grad_dtype
    if gdt == torch.float32 and q.dtype != torch.float32:
        code |= GRAD_F32
    elif gdt != q.dtype:
        raise TypeError("grad_dtype must be the input dtype or torch.float32")
    dq = torch.empty(q.shape, device=q.device, dtype=gdt) if dq is None else dq
    dk = torch.empty(k.shape, device=k.device, dtype=gdt) if dk is None else dk
    dv = torch.empty(v.shape, device=v.device, dtype=gdt) if dv is None else dv
    for t in (dq, dk, dv):
        if t.dtype != gdt:
            raise TypeError("dq, dk, dv must have the gradient dtype")
    return code, dq, dk, dv


def ring_bwd(q, k, v, out, dout, lse, cp, layout=ZIGZAG, causal=True, scale=None,
             dq=None, dk=None, dv=None, workspace=None, grad_dtype=None, tiles_kv_rt=None,
             tiles_q_rt=None, onepass=False):
    """Ring backward on sharded-order tensors; returns (dq, dk, dv).
    grad_dtype=torch.float32 with bf16 inputs writes float32 gradients.
    onepass=True selects the one-pass tensor-core backward (CPATTN_BWD_ONEPASS:
    dQ added by bulk reductions, not bitwise reproducible).
    tiles_kv_rt / tiles_q_rt (int64 [cp, cp] device tensors, zeroed): the
    census of the K/V-major and query-major walks (cpattn_ring_bwd_census)."""
    _need_cuda(q, k, v, out, dout, lse, tiles_kv_rt, tiles_q_rt)
    B, H, Hkv, S, D = _shape(q, k, v)
    code, dq, dk, dv = _grad_args(q, k, v, dq, dk, dv, grad_dtype, onepass)
    need = ring_bwd_workspace_bytes(B, H, Hkv, S, D, code)
    if workspace is None:
        workspace = torch.empty(max(need, 1), device=q.device, dtype=torch.uint8)
    _need_cuda(dq, dk, dv, workspace)
    if tiles_kv_rt is None and tiles_q_rt is None:
        rc = lib().cpattn_ring_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse),
                                   _ptr(dq), _ptr(dk), _ptr(dv), B, H, Hkv, S, D, int(cp),
                                   int(layout), int(bool(causal)), code, _scale(scale),
                                   _ptr(workspace), workspace.numel(), _stream(q))
        _check("cpattn_ring_bwd", rc)
    else:
        for t in (tiles_kv_rt, tiles_q_rt):
            if t is None or t.dtype != torch.int64 or t.numel() < cp * cp:
                raise ValueError("tiles_kv_rt and tiles_q_rt must both be int64 [cp, cp]")
        rc = lib().cpattn_ring_bwd_census(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout),
                                          _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), B, H, Hkv, S,
                                          D, int(cp), int(layout), int(bool(causal)), code,
                                          _scale(scale), _ptr(workspace), workspace.numel(),
                                          _ptr(tiles_kv_rt), _ptr(tiles_q_rt), _stream(q))
        _check("cpattn_ring_bwd_census", rc)
    return dq, dk, dv


def ring_bwd_noalloc(q, k, v, out, dout, lse, cp, layout=ZIGZAG, causal=True, scale=None,
                     dq=None, dk=None, dv=None, grad_dtype=None):
    """cpattn_ring_bwd_noalloc: the ring backward with the library's own fixed
    64 MiB device scratch instead of a workspace, for callers that cannot
    allocate device memory.  Calls that overlap on the GPU race on that scratch."""
    _need_cuda(q, k, v, out, dout, lse)
    B, H, Hkv, S, D = _shape(q, k, v)
    code, dq, dk, dv = _grad_args(q, k, v, dq, dk, dv, grad_dtype)
    _need_cuda(dq, dk, dv)
    rc = lib().cpattn_ring_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout),
                                       _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), B, H, Hkv, S, D,
                                       int(cp), int(layout), int(bool(causal)), code,
                                       _scale(scale), _stream(q))
    _check("cpattn_ring_bwd_noalloc", rc)
    return dq, dk, dv


# ---------------------------------------------------------------------------
# packed documents
# ---------------------------------------------------------------------------

def doc_bounds(cu_seqlens, S, device=None, out=None):
    """Per-position document bounds int32 [S, 2] from offsets cu_seqlens
    (0, strictly increasing, ..., S; a CUDA int32 tensor or anything
    torch.as_tensor takes)."""
    dev = device if device is not None else (
        cu_seqlens.device if torch.is_tensor(cu_seqlens) and cu_seqlens.is_cuda
        else torch.device("cuda", torch.cuda.current_device()))
    cu = cu_seqlens if (torch.is_tensor(cu_seqlens) and cu_seqlens.is_cuda
                        and cu_seqlens.dtype == torch.int32 and cu_seqlens.is_contiguous()) \
        else torch.as_tensor(cu_seqlens, dtype=torch.int32).to(dev).contiguous()
    ndocs = cu.numel() - 1
    bounds = torch.empty((S, 2), device=dev, dtype=torch.int32) if out is None else out
    _need_cuda(bounds)
    rc = lib().cpattn_doc_bounds(_ptr(cu), ndocs, int(S), _ptr(bounds), _stream(cu))
    _check("cpattn_doc_bounds", rc)
    return bounds


def ring_fwd_docs(q, k, v, cp, bounds, layout=ZIGZAG, causal=True, scale=None, out=None,
                  lse=None, tiles_rt=None):
    """Ring forward under the document rule (bounds from doc_bounds)."""
    _need_cuda(q, k, v, bounds)
    B, H, Hkv, S, D = _shape(q, k, v)
    if bounds.dtype != torch.int32 or tuple(bounds.shape) != (S, 2):
        raise ValueError("bounds must be int32 [S, 2] from doc_bounds")
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, S), device=q.device, dtype=torch.float32)
    _need_cuda(out, lse, tiles_rt)
    rc = lib().cpattn_ring_fwd_docs(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Hkv,
                                    S, D, int(cp), int(layout), int(bool(causal)),
                                    _dtype_code(q), _scale(scale), _ptr(bounds), _ptr(tiles_rt),
                                    _stream(q))
    _check("cpattn_ring_fwd_docs", rc)
    return out, lse


def ring_fwd_docs_census(q, k, v, cp, bounds, layout=ZIGZAG, causal=True, scale=None):
    counts = torch.zeros((cp, cp), device=q.device, dtype=torch.int64)
    out, lse = ring_fwd_docs(q, k, v, cp, bounds, layout, causal, scale, tiles_rt=counts)
    return out, lse, counts


def ring_bwd_docs(q, k, v, out, dout, lse, cp, bounds, layout=ZIGZAG, causal=True, scale=None,
                  dq=None, dk=None, dv=None, workspace=None, grad_dtype=None, onepass=False):
    """Ring backward under the document rule; returns (dq, dk, dv)."""
    _need_cuda(q, k, v, out, dout, lse, bounds)
    B, H, Hkv, S, D = _shape(q, k, v)
    if bounds.dtype != torch.int32 or tuple(bounds.shape) != (S, 2):
        raise ValueError("bounds must be int32 [S, 2] from doc_bounds")
    code, dq, dk, dv = _grad_args(q, k, v, dq, dk, dv, grad_dtype, onepass)
    need = ring_bwd_workspace_bytes(B, H, Hkv, S, D, code)
    if workspace is None:
        workspace = torch.empty(max(need, 1), device=q.device, dtype=torch.uint8)
    _need_cuda(dq, dk, dv, workspace)
    rc = lib().cpattn_ring_bwd_docs(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse),
                                    _ptr(dq), _ptr(dk), _ptr(dv), B, H, Hkv, S, D, int(cp),
                                    int(layout), int(bool(causal)), code, _scale(scale),
                                    _ptr(bounds), _ptr(workspace), workspace.numel(), _stream(q))
    _check("cpattn_ring_bwd_docs", rc)
    return dq, dk, dv


def _padded_docs(cu_seqlens, S_real, S, device):
    """Offsets of the real documents plus, when S > S_real, one padding
    document [S_real, S)."""
    cu = [int(x) for x in (cu_seqlens.tolist() if torch.is_tensor(cu_seqlens)
                           else list(cu_seqlens))] if cu_seqlens is not None else [0, S_real]
    if cu[0] != 0 or cu[-1] != S_real:
        raise ValueError(f"cu_seqlens must run from 0 to S={S_real}")
    if S > S_real:
        cu.append(S)
    return doc_bounds(cu, S, device)


# ---------------------------------------------------------------------------
# all-gather K/V schedule
# ---------------------------------------------------------------------------

def _kv_full_shape(q, k_full, v_full):
    B, S, H, D = q.shape
    if k_full.shape != v_full.shape or k_full.shape[0] != B or k_full.shape[1] != S \
            or k_full.shape[3] != D or k_full.dtype != q.dtype or v_full.dtype != q.dtype:
        raise ValueError("k_full, v_full must be [B, S, Hkv, D] of q's dtype")
    return B, H, k_full.shape[2], S, D


def kv_allgather(k, v, cp, layout=ZIGZAG, k_full=None, v_full=None):
    """The all-gather of the sharded K and V on one GPU: every rank's shard
    placed at its natural positions (cpattn_zigzag_unpermute)."""
    return (zigzag_unpermute(k, cp, layout, out=k_full),
            zigzag_unpermute(v, cp, layout, out=v_full))


def allgather_fwd(q, k_full, v_full, cp, layout=ZIGZAG, causal=True, scale=None, bounds=None,
                  out=None, lse=None, tiles_rt=None):
    """Each rank's sharded queries against the whole natural-order K/V in one
    pass (cpattn_allgather_fwd); returns (out, lse) in sharded order."""
    _need_cuda(q, k_full, v_full, bounds)
    B, H, Hkv, S, D = _kv_full_shape(q, k_full, v_full)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, S), device=q.device, dtype=torch.float32)
    _need_cuda(out, lse, tiles_rt)
    rc = lib().cpattn_allgather_fwd(_ptr(q), _ptr(k_full), _ptr(v_full), _ptr(out), _ptr(lse), B,
                                    H, Hkv, S, D, int(cp), int(layout), int(bool(causal)),
                                    _dtype_code(q), _scale(scale), _ptr(bounds), _ptr(tiles_rt),
                                    _stream(q))
    _check("cpattn_allgather_fwd", rc)
    return out, lse


def allgather_bwd(q, k_full, v_full, out, dout, lse, cp, layout=ZIGZAG, causal=True, scale=None,
                  bounds=None, dq=None, dk_full=None, dv_full=None, workspace=None,
                  grad_dtype=None):
    """Backward of the all-gather schedule: dq sharded, dk_full / dv_full in
    natural order summed over every rank's queries."""
    _need_cuda(q, k_full, v_full, out, dout, lse, bounds)
    B, H, Hkv, S, D = _kv_full_shape(q, k_full, v_full)
    code, dq, dk_full, dv_full = _grad_args(q, k_full, v_full, dq, dk_full, dv_full, grad_dtype)
    need = ring_bwd_workspace_bytes(B, H, Hkv, S, D, code)
    if workspace is None:
        workspace = torch.empty(max(need, 1), device=q.device, dtype=torch.uint8)
    _need_cuda(dq, dk_full, dv_full, workspace)
    rc = lib().cpattn_allgather_bwd(_ptr(q), _ptr(k_full), _ptr(v_full), _ptr(out), _ptr(dout),
                                    _ptr(lse), _ptr(dq), _ptr(dk_full), _ptr(dv_full), B, H, Hkv,
                                    S, D, int(cp), int(layout), int(bool(causal)), code,
                                    _scale(scale), _ptr(bounds), _ptr(workspace),
                                    workspace.numel(), _stream(q))
    _check("cpattn_allgather_bwd", rc)
    return dq, dk_full, dv_full


# ---------------------------------------------------------------------------
# Ulysses (all-to-all to head ownership)
# ---------------------------------------------------------------------------

def ulysses_heads(H, Hkv, cp):
    """(query heads, kv heads) per rank after the sequence-to-head all-to-all."""
    hc, grp = H // cp, H // Hkv
    return hc, (hc // grp if hc >= grp else 1)


def ulysses_a2a(x, cp, H, Hkv, layout=ZIGZAG, kv_heads=False, to_seq=False, out=None):
    """One Ulysses all-to-all (cpattn_ulysses_a2a).  Sequence -> head: x
    [B,S,X,D] sharded -> [cp, B, S, nx, D]; head -> sequence: the inverse
    (shared kv heads summed)."""
    _need_cuda(x)
    hc, nkv = ulysses_heads(H, Hkv, cp)
    nx = nkv if kv_heads else hc
    if to_seq:
        _, B, S, _, D = x.shape
        shape = (B, S, Hkv if kv_heads else H, D)
    else:
        B, S, _, D = x.shape
        shape = (cp, B, S, nx, D)
    if out is None:
        out = torch.empty(shape, device=x.device, dtype=x.dtype)
    _need_cuda(out)
    rc = lib().cpattn_ulysses_a2a(_ptr(x), _ptr(out), B, S, H, Hkv, D, int(cp), int(layout),
                                  int(bool(kv_heads)), int(bool(to_seq)), _dtype_code(x),
                                  _stream(x))
    _check("cpattn_ulysses_a2a", rc)
    return out


def ulysses_workspace_bytes(B, H, Hkv, S, D, cp, layout=ZIGZAG, dtype=BF16, backward=False):
    return int(lib().cpattn_ulysses_workspace_bytes(B, H, Hkv, S, D, int(cp), int(layout),
                                                    int(dtype), int(bool(backward))))


def ulysses_fwd(q, k, v, cp, layout=ZIGZAG, causal=True, scale=None, bounds=None, out=None,
                lse=None, workspace=None):
    """The Ulysses variant on sharded-order tensors; returns (out, lse)."""
    _need_cuda(q, k, v, bounds)
    B, H, Hkv, S, D = _shape(q, k, v)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, S), device=q.device, dtype=torch.float32)
    need = ulysses_workspace_bytes(B, H, Hkv, S, D, cp, layout, _dtype_code(q), False)
    if workspace is None:
        workspace = torch.empty(max(need, 1), device=q.device, dtype=torch.uint8)
    _need_cuda(out, lse, workspace)
    rc = lib().cpattn_ulysses_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Hkv, S,
                                  D, int(cp), int(layout), int(bool(causal)), _dtype_code(q),
                                  _scale(scale), _ptr(bounds), _ptr(workspace), workspace.numel(),
                                  _stream(q))
    _check("cpattn_ulysses_fwd", rc)
    return out, lse


def ulysses_bwd(q, k, v, out, dout, lse, cp, layout=ZIGZAG, causal=True, scale=None, bounds=None,
                dq=None, dk=None, dv=None, workspace=None, grad_dtype=None):
    """Backward of the Ulysses variant on sharded-order tensors."""
    _need_cuda(q, k, v, out, dout, lse, bounds)
    B, H, Hkv, S, D = _shape(q, k, v)
    code, dq, dk, dv = _grad_args(q, k, v, dq, dk, dv, grad_dtype)
    need = ulysses_workspace_bytes(B, H, Hkv, S, D, cp, layout, code, True)
    if workspace is None:
        workspace = torch.empty(max(need, 1), device=q.device, dtype=torch.uint8)
    _need_cuda(dq, dk, dv, workspace)
    rc = lib().cpattn_ulysses_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse),
                                  _ptr(dq), _ptr(dk), _ptr(dv), B, H, Hkv, S, D, int(cp),
                                  int(layout), int(bool(causal)), code, _scale(scale),
                                  _ptr(bounds), _ptr(workspace), workspace.numel(), _stream(q))
    _check("cpattn_ulysses_bwd", rc)
    return dq, dk, dv


# ---------------------------------------------------------------------------
# Hierarchical a2a+p2p (all-to-all inside groups, ring across them)
# ---------------------------------------------------------------------------

def hier_a2a(x, cp_a2a, cp_p2p, H, Hkv, layout=ZIGZAG, kv_heads=False, to_seq=False, out=None):
    """The first-level all-to-all (cpattn_hier_a2a).  Sequence -> head: x
    [B,S,X,D] sharded over cp_a2a*cp_p2p ranks -> [cp_a2a, B, S, nx, D], the
    sequence axis in the second level's sharded order; head -> sequence: the
    inverse (shared kv heads summed)."""
    _need_cuda(x)
    hc, nkv = ulysses_heads(H, Hkv, cp_a2a)
    nx = nkv if kv_heads else hc
    if to_seq:
        _, B, S, _, D = x.shape
        shape = (B, S, Hkv if kv_heads else H, D)
    else:
        B, S, _, D = x.shape
        shape = (cp_a2a, B, S, nx, D)
    if out is None:
        out = torch.empty(shape, device=x.device, dtype=x.dtype)
    _need_cuda(out)
    rc = lib().cpattn_hier_a2a(_ptr(x), _ptr(out), B, S, H, Hkv, D, int(cp_a2a), int(cp_p2p),
                               int(layout), int(bool(kv_heads)), int(bool(to_seq)),
                               _dtype_code(x), _stream(x))
    _check("cpattn_hier_a2a", rc)
    return out


def hier_workspace_bytes(B, H, Hkv, S, D, cp_a2a, cp_p2p, layout=ZIGZAG, dtype=BF16,
                         backward=False):
    return int(lib().cpattn_hier_workspace_bytes(B, H, Hkv, S, D, int(cp_a2a), int(cp_p2p),
                                                 int(layout), int(dtype), int(bool(backward))))


def hier_fwd(q, k, v, cp_a2a, cp_p2p, layout=ZIGZAG, causal=True, scale=None, bounds=None,
             out=None, lse=None, workspace=None):
    """The hierarchical schedule on tensors sharded over cp_a2a*cp_p2p ranks;
    returns (out, lse) in the same order."""
    _need_cuda(q, k, v, bounds)
    B, H, Hkv, S, D = _shape(q, k, v)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, S), device=q.device, dtype=torch.float32)
    need = hier_workspace_bytes(B, H, Hkv, S, D, cp_a2a, cp_p2p, layout, _dtype_code(q), False)
    if workspace is None:
        workspace = torch.empty(max(need, 1), device=q.device, dtype=torch.uint8)
    _need_cuda(out, lse, workspace)
    rc = lib().cpattn_hier_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Hkv, S, D,
                               int(cp_a2a), int(cp_p2p), int(layout), int(bool(causal)),
                               _dtype_code(q), _scale(scale), _ptr(bounds), _ptr(workspace),
                               workspace.numel(), _stream(q))
    _check("cpattn_hier_fwd", rc)
    return out, lse


def hier_bwd(q, k, v, out, dout, lse, cp_a2a, cp_p2p, layout=ZIGZAG, causal=True, scale=None,
             bounds=None, dq=None, dk=None, dv=None, workspace=None, grad_dtype=None):
    """Backward of the hierarchical schedule on sharded-order tensors."""
    _need_cuda(q, k, v, out, dout, lse, bounds)
    B, H, Hkv, S, D = _shape(q, k, v)
    code, dq, dk, dv = _grad_args(q, k, v, dq, dk, dv, grad_dtype)
    need = hier_workspace_bytes(B, H, Hkv, S, D, cp_a2a, cp_p2p, layout, code, True)
    if workspace is None:
        workspace = torch.empty(max(need, 1), device=q.device, dtype=torch.uint8)
    _need_cuda(dq, dk, dv, workspace)
    rc = lib().cpattn_hier_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse),
                               _ptr(dq), _ptr(dk), _ptr(dv), B, H, Hkv, S, D, int(cp_a2a),
                               int(cp_p2p), int(layout), int(bool(causal)), code, _scale(scale),
                               _ptr(bounds), _ptr(workspace), workspace.numel(), _stream(q))
    _check("cpattn_hier_bwd", rc)
    return dq, dk, dv


# ---------------------------------------------------------------------------
# census and status
# ---------------------------------------------------------------------------

def tile_counts(S, cp, layout, causal, tile):
    """Closed-form (tiles[cp, cp], pairs[cp, cp]) per (batch, head), host only."""
    import numpy as np
    tiles = np.zeros(cp * cp, dtype=np.uint64)
    pairs = np.zeros(cp * cp, dtype=np.uint64)
    rc = lib().cpattn_tile_counts(int(S), int(cp), int(layout), int(bool(causal)), int(tile),
                                  tiles.ctypes.data_as(ctypes.c_void_p),
                                  pairs.ctypes.data_as(ctypes.c_void_p))
    _check("cpattn_tile_counts", rc)
    return tiles.reshape(cp, cp), pairs.reshape(cp, cp)


def wait_probe(limit_ns, stream=None):
    """cpattn_wait_probe: a bounded device wait that is made to give up."""
    s = ctypes.c_void_p(stream.cuda_stream) if stream is not None else _stream()
    _check("cpattn_wait_probe", lib().cpattn_wait_probe(int(limit_ns), s))


def device_status(stream=None):
    """Synchronises and returns the library status code (0 = OK)."""
    s = ctypes.c_void_p(stream.cuda_stream) if stream is not None else _stream()
    return int(lib().cpattn_device_status(s))


# ---------------------------------------------------------------------------
# natural-order conveniences (the whole hot path)
# ---------------------------------------------------------------------------

def attention(q, k, v, cp, layout=ZIGZAG, causal=True, scale=None):
    """Natural-order in, natural-order out: permute -> ring forward -> unpermute."""
    qs = zigzag_permute(q, cp, layout)
    ks = zigzag_permute(k, cp, layout)
    vs = zigzag_permute(v, cp, layout)
    o, lse = ring_fwd(qs, ks, vs, cp, layout, causal, scale)
    return zigzag_unpermute(o, cp, layout), zigzag_unpermute(lse, cp, layout, seq_dim=2)


def attention_fwd_bwd(q, k, v, dout, cp, layout=ZIGZAG, causal=True, scale=None,
                      grad_dtype=None, onepass=False):
    """Natural order: forward and backward through the ring.  Returns
    (out, lse, dq, dk, dv), all natural order."""
    qs, ks, vs, dos = (zigzag_permute(x, cp, layout) for x in (q, k, v, dout))
    o, lse = ring_fwd(qs, ks, vs, cp, layout, causal, scale)
    dq, dk, dv = ring_bwd(qs, ks, vs, o, dos, lse, cp, layout, causal, scale,
                          grad_dtype=grad_dtype, onepass=onepass)
    un = lambda x: zigzag_unpermute(x, cp, layout)  # noqa: E731
    return un(o), zigzag_unpermute(lse, cp, layout, seq_dim=2), un(dq), un(dk), un(dv)


def attention_docs(q, k, v, cp, cu_seqlens=None, layout=ZIGZAG, causal=True, scale=None):
    """Natural order, any sequence length, packed documents: pads the sequence
    to padded_length (the padding is a document of its own), permutes with
    padding, runs the ring forward under the document rule and drops the
    padding again.  cu_seqlens: document offsets over the real tokens (None:
    one document).  Returns (out, lse) for the real tokens."""
    S_real = q.shape[1]
    S = padded_length(S_real, cp, layout)
    bounds = _padded_docs(cu_seqlens, S_real, S, q.device)
    qs, ks, vs = (zigzag_permute_pad(x, cp, S, layout) for x in (q, k, v))
    o, lse = ring_fwd_docs(qs, ks, vs, cp, bounds, layout, causal, scale)
    return (zigzag_unpermute_pad(o, cp, S_real, layout),
            zigzag_unpermute_pad(lse, cp, S_real, layout, seq_dim=2))


def attention_docs_fwd_bwd(q, k, v, dout, cp, cu_seqlens=None, layout=ZIGZAG, causal=True,
                           scale=None, grad_dtype=None, onepass=False):
    """attention_docs with the backward: dout over the real tokens (the
    padding gets a zero upstream gradient).  Returns (out, lse, dq, dk, dv)
    for the real tokens, natural order."""
    S_real = q.shape[1]
    S = padded_length(S_real, cp, layout)
    bounds = _padded_docs(cu_seqlens, S_real, S, q.device)
    qs, ks, vs, dos = (zigzag_permute_pad(x, cp, S, layout) for x in (q, k, v, dout))
    o, lse = ring_fwd_docs(qs, ks, vs, cp, bounds, layout, causal, scale)
    dq, dk, dv = ring_bwd_docs(qs, ks, vs, o, dos, lse, cp, bounds, layout, causal, scale,
                               grad_dtype=grad_dtype, onepass=onepass)
    un = lambda x: zigzag_unpermute_pad(x, cp, S_real, layout)  # noqa: E731
    return (un(o), zigzag_unpermute_pad(lse, cp, S_real, layout, seq_dim=2), un(dq), un(dk),
            un(dv))


def attention_allgather_fwd_bwd(q, k, v, dout, cp, layout=ZIGZAG, causal=True, scale=None,
                                grad_dtype=None):
    """Natural order in and out, through the all-gather schedule: shard Q,
    dO (and K, V as the ranks hold them), all-gather K/V, attend, backward,
    reduce-scatter dK/dV to their owners, unshard.  Returns (out, lse, dq,
    dk, dv) in natural order."""
    qs, ks, vs, dos = (zigzag_permute(x, cp, layout) for x in (q, k, v, dout))
    kf, vf = kv_allgather(ks, vs, cp, layout)
    o, lse = allgather_fwd(qs, kf, vf, cp, layout, causal, scale)
    dq, dkf, dvf = allgather_bwd(qs, kf, vf, o, dos, lse, cp, layout, causal, scale,
                                 grad_dtype=grad_dtype)
    dks, dvs = zigzag_permute(dkf, cp, layout), zigzag_permute(dvf, cp, layout)
    un = lambda x: zigzag_unpermute(x, cp, layout)  # noqa: E731
    return un(o), zigzag_unpermute(lse, cp, layout, seq_dim=2), un(dq), un(dks), un(dvs)


def attention_ulysses_fwd_bwd(q, k, v, dout, cp, layout=ZIGZAG, causal=True, scale=None,
                              grad_dtype=None):
    """Natural order in and out through the Ulysses variant: shard, all-to-all
    to head owners, attend, backward, all-to-all back, unshard.  Returns
    (out, lse, dq, dk, dv) in natural order."""
    qs, ks, vs, dos = (zigzag_permute(x, cp, layout) for x in (q, k, v, dout))
    o, lse = ulysses_fwd(qs, ks, vs, cp, layout, causal, scale)
    dq, dk, dv = ulysses_bwd(qs, ks, vs, o, dos, lse, cp, layout, causal, scale,
                             grad_dtype=grad_dtype)
    un = lambda x: zigzag_unpermute(x, cp, layout)  # noqa: E731
    return un(o), zigzag_unpermute(lse, cp, layout, seq_dim=2), un(dq), un(dk), un(dv)


def attention_host_workspace_bytes(B, H, Hkv, S, D, cp, layout=ZIGZAG, dtype=BF16,
                                   backward=True) -> int:
    return int(lib().cpattn_attention_host_workspace_bytes(B, H, Hkv, S, D, int(cp), int(layout),
                                                           int(dtype), int(bool(backward))))


def attention_host_parts(B, H, Hkv, S, D) -> int:
    """The number of head parts attention_host takes when parts=0."""
    return int(lib().cpattn_attention_host_parts(B, H, Hkv, S, D))


def _host_prepare(q, k, v, dout, out, lse, dq, dk, dv, grad_dtype, device, name, onepass=False):
    """Shared marshalling of the host-to-host calls: checks, dtype code,
    output tensors (pinned when the inputs are)."""
    if q.is_cuda or k.is_cuda or v.is_cuda:
        raise ValueError(f"{name} takes host (CPU) tensors")
    for t in (q, k, v, dout):
        if t is not None and not t.is_contiguous():
            raise ValueError("tensor must be contiguous")
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    B, S, H, D = q.shape
    code = _dtype_code(q)
    backward = dout is not None
    gdt = q.dtype if grad_dtype is None else grad_dtype
    if backward and gdt == torch.float32 and q.dtype != torch.float32:
        code |= GRAD_F32
    if backward and onepass:
        code |= ONEPASS
    pin = q.is_pinned()

    def host(shape, dtype, t):
        return torch.empty(shape, dtype=dtype, pin_memory=pin) if t is None else t
    out = host(q.shape, q.dtype, out)
    lse = host((B, H, S), torch.float32, lse)
    if backward:
        dq = host(q.shape, gdt, dq)
        dk = host(k.shape, gdt, dk)
        dv = host(v.shape, gdt, dv)
    return dev, code, backward, (out, lse, dq, dk, dv)


def attention_host(q, k, v, dout, cp, layout=ZIGZAG, causal=True, scale=None, out=None,
                   lse=None, dq=None, dk=None, dv=None, grad_dtype=None, workspace=None,
                   device=None, stream=None, parts=0, onepass=False):
    """cpattn_attention_host: natural-order CPU tensors (pinned for
    asynchronous copies) in and out, the whole path on the GPU in between,
    the heads in `parts` pipelined groups (0: the library's choice).
    dout None: forward only.  Returns (out, lse) or (out, lse, dq, dk, dv) as
    CPU tensors; they are complete once the stream has been synchronised."""
    dev, code, backward, res = _host_prepare(q, k, v, dout, out, lse, dq, dk, dv, grad_dtype,
                                             device, "attention_host", onepass)
    B, S, H, D = q.shape
    Hkv = k.shape[2]
    need = attention_host_workspace_bytes(B, H, Hkv, S, D, cp, layout, code, backward)
    if workspace is None:
        workspace = torch.empty(max(need, 1), device=dev, dtype=torch.uint8)
    st = ctypes.c_void_p((stream or torch.cuda.current_stream(dev)).cuda_stream)
    rc = lib().cpattn_attention_host(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), *map(_ptr, res), B, H,
                                     Hkv, S, D, int(cp), int(layout), int(bool(causal)), code,
                                     _scale(scale), int(parts), _ptr(workspace), workspace.numel(),
                                     st)
    _check("cpattn_attention_host", rc)
    return res if backward else res[:2]


def attention_host_docs_workspace_bytes(B, H, Hkv, S, D, cp, layout=ZIGZAG, dtype=BF16,
                                        backward=True) -> int:
    return int(lib().cpattn_attention_host_docs_workspace_bytes(B, H, Hkv, S, D, int(cp),
                                                                int(layout), int(dtype),
                                                                int(bool(backward))))


def attention_host_docs(q, k, v, dout, cp, cu_seqlens=None, layout=ZIGZAG, causal=True,
                        scale=None, out=None, lse=None, dq=None, dk=None, dv=None,
                        grad_dtype=None, workspace=None, device=None, stream=None, parts=0,
                        onepass=False):
    """cpattn_attention_host_docs: attention_host for packed documents and any
    sequence length.  cu_seqlens: document offsets over the S tokens (a
    sequence of ints, 0 ... S), None for one document.  Returns (out, lse) or
    (out, lse, dq, dk, dv) as CPU tensors over the S real tokens."""
    dev, code, backward, res = _host_prepare(q, k, v, dout, out, lse, dq, dk, dv, grad_dtype,
                                             device, "attention_host_docs", onepass)
    B, S, H, D = q.shape
    Hkv = k.shape[2]
    need = attention_host_docs_workspace_bytes(B, H, Hkv, S, D, cp, layout, code, backward)
    if workspace is None:
        workspace = torch.empty(max(need, 1), device=dev, dtype=torch.uint8)
    cu_arr, ndocs = None, 0
    if cu_seqlens is not None:
        cu_list = [int(x) for x in cu_seqlens]
        cu_arr, ndocs = (ctypes.c_int32 * len(cu_list))(*cu_list), len(cu_list) - 1
    st = ctypes.c_void_p((stream or torch.cuda.current_stream(dev)).cuda_stream)
    rc = lib().cpattn_attention_host_docs(
        _ptr(q), _ptr(k), _ptr(v), _ptr(dout), *map(_ptr, res), B, H, Hkv, S, D, int(cp),
        int(layout), int(bool(causal)), code, _scale(scale),
        ctypes.cast(cu_arr, ctypes.c_void_p) if cu_arr is not None else None, ndocs, int(parts),
        _ptr(workspace), workspace.numel(), st)
    _check("cpattn_attention_host_docs", rc)
    return res if backward else res[:2]


def attention_hier_fwd_bwd(q, k, v, dout, cp_a2a, cp_p2p, layout=ZIGZAG, causal=True,
                           scale=None, grad_dtype=None):
    """Natural order in and out through the hierarchical schedule: shard over
    cp_a2a*cp_p2p ranks, all-to-all inside groups, second-level ring,
    backward, all-to-all back, unshard.  Returns (out, lse, dq, dk, dv)."""
    cp = cp_a2a * cp_p2p
    qs, ks, vs, dos = (zigzag_permute(x, cp, layout) for x in (q, k, v, dout))
    o, lse = hier_fwd(qs, ks, vs, cp_a2a, cp_p2p, layout, causal, scale)
    dq, dk, dv = hier_bwd(qs, ks, vs, o, dos, lse, cp_a2a, cp_p2p, layout, causal, scale,
                          grad_dtype=grad_dtype)
    un = lambda x: zigzag_unpermute(x, cp, layout)  # noqa: E731
    return un(o), zigzag_unpermute(lse, cp, layout, seq_dim=2), un(dq), un(dk), un(dv)
