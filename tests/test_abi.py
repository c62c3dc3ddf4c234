"""The C ABI without a GPU: libpfa builds, loads, exports every declared symbol, and rejects
bad arguments before it touches a device."""
import ctypes
import os
import re

import pytest

from precision_flash_attention_gb300 import _lib, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "pfa.h")


@pytest.fixture(scope="module")
def lib():
    build.build_library()
    return _lib.load()


def _declared():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pfa_[a-z_]+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert sorted(_lib.EXPORTS) == _declared()


def test_binding_constants_match_the_header():
    # Every option flag, the tie-histogram size and every status code the binding uses
    # is the value include/pfa.h gives it.
    text = re.sub(r"/\*.*?\*/", "", open(HEADER, encoding="utf-8").read(), flags=re.S)
    defines = {n: int(v) for n, v in re.findall(r"#define\s+PFA_([A-Z0-9_]+)\s+(\d+)u?\b", text)}
    for name in ("FWD_UNFUSED_BF16_PV", "FWD_PBAR_E4M3", "FWD_PBAR_MXFP4", "FWD_PAIR_CTA",
                 "BWD_DQ_DETERMINISTIC", "BWD_DQ_SPLIT", "BWD_WORKSPACE_ZEROED", "TIE_BINS",
                 "DEVERR_TIMEOUT", "DEVERR_SMEM_ALIGN"):
        assert getattr(_lib, name) == defines[name], name
    status = {int(v): "PFA_" + n for n, v in re.findall(r"\bPFA_((?:OK|ERR_[A-Z_]+))\s*=\s*(-?\d+)", text)}
    assert status == _lib.STATUS_NAMES


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings(lib):
    for code, name in _lib.STATUS_NAMES.items():
        assert lib.pfa_status_string(code).decode().startswith(name)
    assert lib.pfa_status_string(12345).decode() == "PFA_ERR_UNKNOWN"


def test_workspace_bytes(lib):
    assert lib.pfa_bwd_workspace_bytes(8, 12, 1024, 64) == 8 * 12 * 1024 * 64 * 4
    assert lib.pfa_bwd_workspace_bytes(1, 1, 1, 128) == 512
    assert lib.pfa_bwd_workspace_bytes(1, 1, 1, 96) == 0
    assert lib.pfa_bwd_workspace_bytes(0, 1, 16, 64) == 0
    assert lib.pfa_bwd_workspace_bytes(4096, 64, 8192, 128) == 0  # over 2^31 elements


A = 1 << 20  # a fake, 16-byte aligned "device" address; never dereferenced on these paths


def _no_device():
    """Calls that pass validation would launch kernels on the fake addresses: they are
    made only where no CUDA device exists, so they fail on the device lookup."""
    import torch
    return not torch.cuda.is_available()


def _fwd(lib, **kw):
    args = dict(q=A, k=A, v=A, o=A, lse=A, B=1, Hq=2, Hkv=1, N=64, d=64, causal=0, scale=0.125,
                mode=1, beta=2.0, eps=1e-3, counters=None, stream=None)
    args.update(kw)
    return lib.pfa_attn_fwd(*args.values())


def test_fwd_argument_errors(lib):
    inv, mis = -1, -2
    assert _fwd(lib, q=None) == inv
    assert _fwd(lib, lse=None) == inv
    assert _fwd(lib, N=0) == inv
    assert _fwd(lib, d=96) == inv
    assert _fwd(lib, Hq=3, Hkv=2) == inv
    assert _fwd(lib, mode=3) == inv
    assert _fwd(lib, mode=-1) == inv
    assert _fwd(lib, beta=1.0) == inv            # the fix needs beta > 1
    assert _fwd(lib, beta=float("nan")) == inv
    assert _fwd(lib, eps=-1e-3) == inv
    assert _fwd(lib, eps=float("inf")) == inv
    assert _fwd(lib, scale=0.0) == inv
    assert _fwd(lib, scale=float("nan")) == inv
    assert _fwd(lib, q=A + 8) == mis
    assert _fwd(lib, counters=A + 4) == mis
    assert _fwd(lib, mode=0, eps=-1.0, counters=A) == inv
    # beta is not checked in mode 0/2, eps not in mode 0 without counters: the call gets
    # past validation and fails only on the missing device.
    if _no_device():
        assert _fwd(lib, mode=0, beta=0.5, eps=-1.0) not in (inv, mis)


def test_other_entry_points_validate(lib):
    inv, mis = -1, -2
    assert lib.pfa_attn_delta(None, A, A, 1, 1, 64, 64, None) == inv
    assert lib.pfa_attn_delta(A, A, A + 4, 1, 1, 64, 64, None) == mis
    assert lib.pfa_attn_delta(A, A, A, 1, 1, 64, 32, None) == inv
    assert lib.pfa_attn_delta_alt(A, A, A, A, A, A, 1, 2, 1, 64, 64, 1, -1.0, None) == inv
    assert lib.pfa_attn_delta_alt(A, A, A, A, A, None, 1, 2, 1, 64, 64, 1, 0.1, None) == inv
    args = [A] * 10 + [1, 2, 1, 64, 64, 1, 0.125, None]
    bad = list(args)
    bad[9] = None  # no workspace
    assert lib.pfa_attn_bwd(*bad) == inv
    bad = list(args)
    bad[6] = A + 2
    assert lib.pfa_attn_bwd(*bad) == mis
    bad = list(args)
    bad[12] = 3  # H_kv does not divide H_q
    assert lib.pfa_attn_bwd(*bad) == inv


def test_without_a_device_calls_fail_cleanly(lib):
    if not _no_device():
        pytest.skip("a device is present")
    assert _fwd(lib) in (-3, -4)
    assert lib.pfa_device_error(0) in (-3, -4)


def test_accumulate_and_noalloc_entry_points_validate(lib):
    inv, mis, too_large = -1, -2, -6
    # pfa_attn_bwd_accum: the same checks as pfa_attn_bwd, before any device call.
    args = [A] * 9 + [1, 2, 1, 64, 64, 1, 0.125, None]
    for i in range(9):
        bad = list(args)
        bad[i] = None
        assert lib.pfa_attn_bwd_accum(*bad) == inv, i
    bad = list(args)
    bad[6] = A + 4                       # the FP32 accumulator, misaligned
    assert lib.pfa_attn_bwd_accum(*bad) == mis
    bad = list(args)
    bad[11] = 3                          # H_kv does not divide H_q
    assert lib.pfa_attn_bwd_accum(*bad) == inv
    bad = list(args)
    bad[13] = 32                         # d not in {64, 128}
    assert lib.pfa_attn_bwd_accum(*bad) == inv
    bad = list(args)
    bad[15] = float("inf")               # scale
    assert lib.pfa_attn_bwd_accum(*bad) == inv
    # pfa_attn_bwd_noalloc: sizes are checked first, then the fixed buffer's limit.
    nargs = [A] * 9 + [1, 2, 1, 64, 64, 1, 0.125, None]
    bad = list(nargs)
    bad[13] = 96
    assert lib.pfa_attn_bwd_noalloc(*bad) == inv
    bad = list(nargs)
    bad[9], bad[10], bad[11], bad[12] = 8, 16, 8, 8192   # 8*16*8192*64 values > 8,388,608
    assert lib.pfa_attn_bwd_noalloc(*bad) == too_large
    if _no_device():
        bad[12] = 1024                                   # 8*16*1024*64 = 8,388,608: fits
        assert lib.pfa_attn_bwd_noalloc(*bad) != too_large


def test_bwd_ex_validates(lib):
    inv, mis = -1, -2
    args = [A] * 10 + [1, 2, 1, 64, 64, 1, 0.125, 0, None]
    bad = list(args)
    bad[17] = 8                          # an unknown flag bit
    assert lib.pfa_attn_bwd_ex(*bad) == inv
    bad = list(args)
    bad[17], bad[9] = 4, None            # a zeroed workspace is still a workspace
    assert lib.pfa_attn_bwd_ex(*bad) == inv
    bad = list(args)
    bad[17], bad[6] = 1, None            # the query-outer pass needs dq
    assert lib.pfa_attn_bwd_ex(*bad) == inv
    bad = list(args)
    bad[17], bad[6] = 3, A + 2           # misaligned dq
    assert lib.pfa_attn_bwd_ex(*bad) == mis
    bad = list(args)
    bad[9] = None                        # flags 0 is pfa_attn_bwd: the workspace is required
    assert lib.pfa_attn_bwd_ex(*bad) == inv
    if _no_device():
        bad = list(args)
        bad[17], bad[9] = 2, None        # with the query-outer pass dq_accum may be NULL
        assert lib.pfa_attn_bwd_ex(*bad) not in (inv, mis)


def test_fwd_ex_validates(lib):
    inv, mis = -1, -2
    args = dict(q=A, k=A, v=A, o=A, lse=A, B=1, Hq=2, Hkv=1, N=64, d=64, causal=0, scale=0.125,
                mode=0, beta=2.0, eps=1e-3, counters=None, monitor=None, flags=0, stream=None)

    def call(**kw):
        a = dict(args)
        a.update(kw)
        return lib.pfa_attn_fwd_ex(*a.values())

    assert call(flags=16) == inv                      # an unknown flag bit
    assert call(flags=2 | 4) == inv                   # both narrow Pbar formats at once
    # The CTA pairing is built for the fused d = 128 path only.
    assert call(flags=8) == -3
    assert call(flags=8, d=128, monitor=A) == -3
    assert call(flags=8 | 2, d=128) == -3
    assert call(monitor=A + 4) == mis                 # the monitor must be 8-byte aligned
    assert call(monitor=A, eps=-1.0) == inv           # the monitor needs a valid eps
    assert call(q=None) == inv
    if _no_device():
        for fl in (1, 2, 4, 1 | 2):
            assert call(flags=fl, d=128) == -3        # the study variants are d = 64 only
            assert call(flags=fl) not in (inv, mis)


def test_delta_zero_validates(lib):
    inv, mis = -1, -2
    args = [A, A, A, A, 1, 2, 64, 64, None]
    assert lib.pfa_attn_delta_zero(*args[:3], None, *args[4:]) == inv   # the workspace is required
    assert lib.pfa_attn_delta_zero(*args[:3], A + 4, *args[4:]) == mis  # misaligned workspace
    assert lib.pfa_attn_delta_zero(*args[:4], 1, 2, 64, 96, None) == inv  # d not 64 or 128
