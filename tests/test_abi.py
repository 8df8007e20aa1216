"""Host-side checks of libcpattn that need no GPU: the library loads, exports
every entry point include/cpattn.h declares, validates arguments before any
launch, and its closed-form work census equals the oracle's enumeration."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import context_causal_attention_zigzag_gb300 as cp_attn
from context_causal_attention_zigzag_gb300 import _binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "cpattn.h")


def declared_entry_points():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"CPATTN_API\s+[\w\s\*]*?\b(cpattn_\w+)\s*\(", text)))


def test_library_loads_and_exports_every_declared_symbol():
    names = declared_entry_points()
    assert len(names) >= 13
    lib = cp_attn.lib()
    for n in names:
        assert hasattr(lib, n), n
        assert n in _binding.SIGNATURES, f"{n} has no ctypes signature"
    assert set(_binding.SIGNATURES) == set(names)


def declared_parameter_counts():
    """name -> number of parameters, read from the CPATTN_API declarations."""
    text = open(HEADER).read()
    out = {}
    for m in re.finditer(r"CPATTN_API\s+[\w\s\*]*?\b(cpattn_\w+)\s*\(([^;]*?)\)\s*;", text,
                         re.S):
        params = m.group(2).strip()
        out[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_ctypes_signatures_match_header_parameter_counts():
    counts = declared_parameter_counts()
    assert set(counts) == set(_binding.SIGNATURES)
    for name, (_, args) in _binding.SIGNATURES.items():
        assert len(args) == counts[name], (name, len(args), counts[name])


def test_status_strings():
    for code in (0, -1, -2, -3, -4, -5, 7):
        assert isinstance(cp_attn.status_string(code), str)
    assert cp_attn.status_string(-4) != cp_attn.status_string(-3)


@pytest.mark.parametrize("layout", [oracle.ZIGZAG, oracle.CONTIGUOUS])
@pytest.mark.parametrize("causal", [True, False])
def test_tile_census_closed_form_equals_enumeration(layout, causal):
    for cp in (1, 2, 3, 4, 8, 16):
        for T in (1, 4, 64):
            for n in (1, 2, 5):
                per = 2 if layout == oracle.ZIGZAG else 1
                S = cp * per * n * T
                tiles, pairs = cp_attn.tile_counts(S, cp, layout, causal, T)
                want_pairs = S <= 4096
                ot, op = oracle.tile_counts(S, cp, layout, causal, T, pairs=want_pairs)
                np.testing.assert_array_equal(tiles, ot)
                if want_pairs:
                    np.testing.assert_array_equal(pairs, op)
                if causal:
                    assert int(pairs.sum()) == S * (S + 1) // 2
                else:
                    assert int(pairs.sum()) == S * S


def test_tile_census_full_size_workloads():
    # The per-step tile table at T = 128 for the named workloads, closed form
    # vs enumeration, and the zigzag balance (max/mean per step == 1).
    cases = [(8192, 4, oracle.ZIGZAG, True), (8192, 4, oracle.CONTIGUOUS, True),
             (32768, 8, oracle.ZIGZAG, True), (16384, 4, oracle.CONTIGUOUS, False),
             (131072, 16, oracle.ZIGZAG, True)]
    for S, cp, layout, causal in cases:
        tiles, _ = cp_attn.tile_counts(S, cp, layout, causal, 128)
        ot, _ = oracle.tile_counts(S, cp, layout, causal, 128)
        np.testing.assert_array_equal(tiles, ot)
        if layout == oracle.ZIGZAG:
            per_step = tiles.astype(np.float64)
            assert np.all(per_step.max(axis=0) == per_step.mean(axis=0))


def test_plan():
    path, tile = cp_attn.plan(1, 2, 2, 256, 64, 2, cp_attn.ZIGZAG, True, cp_attn.F32)
    assert path == cp_attn.PATH_SIMT and tile == 64
    for w in [(1, 32, 32, 8192, 128, 4), (2, 32, 8, 32768, 128, 8), (1, 32, 8, 131072, 128, 16)]:
        path, tile = cp_attn.plan(*w, cp_attn.ZIGZAG, True, cp_attn.BF16)
        assert path in (cp_attn.PATH_SIMT, cp_attn.PATH_TCGEN05)
        assert tile == (128 if path == cp_attn.PATH_TCGEN05 else 64)


def test_invalid_arguments_rejected_before_launch():
    lib = cp_attn.lib()
    null = ctypes.c_void_p(0)
    fake = ctypes.c_void_p(0x1000)
    E = _binding.ERR_INVALID_ARG
    fwd = lib.cpattn_ring_fwd
    # (B, H, Hkv, S, D, cp, layout, causal, dtype)
    good = [1, 4, 2, 64, 64, 2, 1, 1, 1]
    bad_cases = [
        [1, 4, 3, 64, 64, 2, 1, 1, 1],   # H % Hkv
        [1, 4, 2, 60, 64, 4, 1, 1, 1],   # S % (2 cp)
        [1, 4, 2, 64, 96, 2, 1, 1, 1],   # D
        [1, 4, 2, 64, 64, 0, 1, 1, 1],   # cp
        [1, 4, 2, 64, 64, 2, 7, 1, 1],   # layout
        [1, 4, 2, 64, 64, 2, 1, 1, 9],   # dtype
        [-1, 4, 2, 64, 64, 2, 1, 1, 1],  # B
    ]
    for args in bad_cases:
        assert fwd(fake, fake, fake, fake, fake, *args, 0.0, null) == E, args
    # null pointers with a valid shape
    assert fwd(null, fake, fake, fake, fake, *good, 0.0, null) == E
    # misaligned pointer
    assert fwd(ctypes.c_void_p(0x1002), fake, fake, fake, fake, *good, 0.0, null) == E
    # empty problem is a no-op success
    assert fwd(null, null, null, null, null, 0, 4, 2, 64, 64, 2, 1, 1, 1, 0.0, null) == 0
    # ring step out of range
    assert lib.cpattn_ring_fwd_step(fake, fake, fake, *good, 0.0, 2, fake, fake, null) == E
    # permute: bad S, overlap
    assert lib.cpattn_zigzag_permute(fake, ctypes.c_void_p(0x9000), 1, 60, 16, 4, 1, null) == E
    assert lib.cpattn_zigzag_permute(fake, ctypes.c_void_p(0x1010), 1, 64, 16, 4, 1, null) == E
    # merge: D
    assert lib.cpattn_lse_merge(fake, fake, fake, fake, fake, fake, 1, 8, 2, 32, null) == E
    # backward: workspace too small / missing
    need = lib.cpattn_ring_bwd_workspace_bytes(1, 4, 2, 64, 64, 1)
    assert need >= 4 * 64 * 4 * 64
    args9 = [fake] * 9
    assert lib.cpattn_ring_bwd(*args9, *good, 0.0, null, need, null) == _binding.ERR_WORKSPACE
    assert lib.cpattn_ring_bwd(*args9, *good, 0.0, fake, need - 1, null) == _binding.ERR_WORKSPACE
    assert lib.cpattn_ring_bwd(*args9, *[1, 4, 3] + good[3:], 0.0, fake, need, null) == E
    # census needs its output
    assert lib.cpattn_ring_fwd_census(fake, fake, fake, fake, fake, *good, 0.0, null, null) == E
    # closed-form census: chunk length not a multiple of the tile
    arr = (ctypes.c_uint64 * 16)()
    assert lib.cpattn_tile_counts(96, 4, 1, 1, 8, arr, None) == E
    # documents: bounds missing or misaligned, document count out of range
    assert lib.cpattn_ring_fwd_docs(fake, fake, fake, fake, fake, *good, 0.0, null, null,
                                    null) == E
    assert lib.cpattn_ring_fwd_docs(fake, fake, fake, fake, fake, *good, 0.0,
                                    ctypes.c_void_p(0x1004), null, null) == E
    assert lib.cpattn_ring_bwd_docs(*args9, *good, 0.0, null, fake, need, null) == E
    assert lib.cpattn_doc_bounds(fake, 0, 64, fake, null) == E
    assert lib.cpattn_doc_bounds(fake, 65, 64, fake, null) == E
    assert lib.cpattn_doc_bounds(null, 2, 64, fake, null) == E
    assert lib.cpattn_doc_bounds(fake, 2, 64, ctypes.c_void_p(0x1004), null) == E
    # padded permute: real length above the padded one
    assert lib.cpattn_zigzag_permute_pad(fake, ctypes.c_void_p(0x90000), 1, 65, 64, 16, 4, 1,
                                         null) == E
    # host path: parts must divide Hkv and lie in 0..8; workspace checked next
    host = lib.cpattn_attention_host
    hneed = lib.cpattn_attention_host_workspace_bytes(*good, 1)
    assert hneed > 0
    for parts in (3, -1, 9):
        assert host(*args9, *good, 0.0, parts, fake, hneed, null) == E, parts
    assert host(*args9, *good, 0.0, 2, null, hneed, null) == _binding.ERR_WORKSPACE
    assert host(*args9, *good, 0.0, 2, ctypes.c_void_p(0x1010), hneed, null) == \
        _binding.ERR_WORKSPACE  # not 256-byte aligned


def test_host_docs_rejects_bad_offsets_before_any_copy():
    lib = cp_attn.lib()
    null = ctypes.c_void_p(0)
    fake = ctypes.c_void_p(0x1000)
    E = _binding.ERR_INVALID_ARG
    args9 = [fake] * 9
    shape = [1, 4, 2, 100, 64, 2, 1, 1, 1]  # S = 100 real tokens, padded on the device
    need = lib.cpattn_attention_host_docs_workspace_bytes(*shape, 1)
    assert need > 0
    for cu in ([0, 50, 40, 100], [0, 50, 99], [1, 50, 100], [0, 100, 100]):
        arr = (ctypes.c_int32 * len(cu))(*cu)
        rc = lib.cpattn_attention_host_docs(*args9, *shape, 0.0, ctypes.cast(arr, ctypes.c_void_p),
                                            len(cu) - 1, 0, fake, need, null)
        assert rc == E, cu
    assert lib.cpattn_attention_host_docs(*args9, *shape, 0.0, null, 0, 3, fake, need, null) == E


def test_host_parts_choice():
    lib = cp_attn.lib()
    assert lib.cpattn_attention_host_parts(1, 32, 8, 131072, 128) == 8   # 1 GiB of Q, Hkv 8
    assert lib.cpattn_attention_host_parts(1, 32, 8, 16384, 128) == 2    # 128 MiB of Q
    assert lib.cpattn_attention_host_parts(1, 32, 2, 131072, 128) == 2   # Hkv 2
    assert lib.cpattn_attention_host_parts(1, 32, 1, 131072, 128) == 1   # one kv head
    assert lib.cpattn_attention_host_parts(1, 4, 2, 2048, 128) == 1      # small
    assert lib.cpattn_attention_host_parts(1, 4, 3, 2048, 128) == 1      # invalid shape


@pytest.mark.parametrize("layout", [_binding.CONTIGUOUS, _binding.ZIGZAG])
def test_padded_length(layout):
    # The smallest length >= S whose chunks are whole 256-token query pairs.
    per = 2 if layout == _binding.ZIGZAG else 1
    for cp in (1, 2, 3, 4, 8, 16):
        unit = cp * per * 256
        for S in (0, 1, 255, unit - 1, unit, unit + 1, 5 * unit + 7, 131072):
            got = cp_attn.padded_length(S, cp, layout)
            assert got >= S and got % unit == 0 and got - S < unit, (S, cp, got)
    assert cp_attn.lib().cpattn_padded_length(-1, 2, layout) == -1
    assert cp_attn.lib().cpattn_padded_length(10, 0, layout) == -1
    assert cp_attn.lib().cpattn_padded_length(10, 2, 5) == -1


def test_balance_report_closed_form():
    # Zigzag: every ring step perfectly balanced; contiguous: step t has
    # max/mean = cp/(cp-t) and lockstep efficiency 0.575 / 0.534 / 0.516 for
    # the S=8192 cp=4, S=32768 cp=8 and S=131072 cp=16 workloads.
    from context_causal_attention_zigzag_gb300 import balance
    for S, cp, eff in ((8192, 4, 0.575), (32768, 8, 0.534), (131072, 16, 0.516)):
        r = balance.report(S=S, cp=cp, run_kernel=False)
        assert r["zigzag"]["closed_form"]["worst_step_max_over_mean"] == 1.0
        assert r["zigzag"]["closed_form"]["lockstep_efficiency"] == 1.0
        ratios = r["contiguous"]["closed_form"]["max_over_mean_per_step"]
        assert np.allclose(ratios, [cp / (cp - t) for t in range(cp)])
        assert abs(r["contiguous"]["closed_form"]["lockstep_efficiency"] - eff) < 5e-4
