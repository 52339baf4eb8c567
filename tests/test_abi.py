"""The C-ABI library builds, loads without a GPU, exports every declared entry point, and its
host-side argument checks reject bad calls before touching CUDA (CPU only)."""
import ctypes
import os
import re

import pytest

import exact_attention_13_gb300 as ea
from exact_attention_13_gb300 import _build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "exact_attention.h")


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"FA_API\s+[\w\s\*]+?\b(fa_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return ea.lib()


def test_header_declares_the_entry_points():
    names = declared_functions()
    assert "fa_fwd" in names and "fa_fwd_ex" in names
    assert set(names) == set(ea.SIGNATURES), (names, sorted(ea.SIGNATURES))


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings_and_version(lib):
    assert ea.version() == 100
    for code in range(6):
        s = lib.fa_status_string(code).decode()
        assert s and s != "unknown status"
    assert lib.fa_status_string(99).decode() == "unknown status"


FAKE = 0x10000  # never dereferenced: each call below fails its host-side checks first


@pytest.mark.parametrize("args,want", [
    ((0, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 128, 0.1, 0, 0), ea.FA_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, 0, 1, 1, 128, 128, 0.1, 0, 0), ea.FA_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 0, 1, 128, 128, 0.1, 0, 0), ea.FA_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, -5, 128, 0.1, 0, 0), ea.FA_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 128, -0.5, 0, 0), ea.FA_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 128, float("inf"), 0, 0), ea.FA_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 128, 0.1, 0, 3), ea.FA_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 96, 0.1, 0, 0), ea.FA_ERR_UNSUPPORTED),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 256, 0.1, 0, 0), ea.FA_ERR_UNSUPPORTED),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 256, 256, 128, 128, 0.1, 0, 0), ea.FA_ERR_UNSUPPORTED),
    ((FAKE + 8, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 128, 0.1, 0, 0), ea.FA_ERR_MISALIGNED),
    ((FAKE, FAKE, FAKE, FAKE + 2, FAKE, 1, 1, 128, 128, 0.1, 1, 0), ea.FA_ERR_MISALIGNED),
    ((FAKE, FAKE, FAKE, FAKE, FAKE + 1, 1, 1, 128, 64, 0.1, 1, 1), ea.FA_ERR_MISALIGNED),
])
def test_host_checks(lib, args, want):
    assert ea.fa_fwd(*args, None) == want


def test_bad_descales_rejected(lib):
    for ds in ((0.0, 1.0, 1.0), (1.0, float("nan"), 1.0), (1.0, 1.0, -2.0)):
        rc = ea.fa_fwd_ex(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 128, 0.1, 0,
                          ea.FA_DTYPE_FP8_E4M3, ds, None, None)
        assert rc == ea.FA_ERR_INVALID_ARG


def test_debug_exp2_checks(lib):
    assert lib.fa_debug_exp2(None, None, 10, 0, None) == ea.FA_ERR_INVALID_ARG
    assert lib.fa_debug_exp2(FAKE, FAKE, 10, 2, None) == ea.FA_ERR_INVALID_ARG
    assert lib.fa_debug_exp2(FAKE, FAKE, 0, 0, None) == ea.FA_OK


def test_split_workspace_bytes(lib):
    assert ea.split_workspace_bytes(1, 2, 300, 128, 3) == (3 * 2 * 300 * 129 * 4 + 255) // 256 * 256
    assert ea.split_workspace_bytes(1, 1, 1, 64, 1) == 512  # 65 floats -> 260 B -> 512
    for bad in ((0, 1, 8, 64, 2), (1, 1, 8, 96, 2), (1, 1, 8, 64, 0), (1, 1, 8, 64, 17)):
        assert ea.split_workspace_bytes(*bad) == 0


@pytest.mark.parametrize("splits,ws,nbytes,want", [
    (0, FAKE, 1 << 30, ea.FA_ERR_INVALID_ARG),
    (17, FAKE, 1 << 30, ea.FA_ERR_INVALID_ARG),
    (2, 0, 1 << 30, ea.FA_ERR_INVALID_ARG),
    (2, FAKE, 1024, ea.FA_ERR_INVALID_ARG),
    (2, FAKE + 4, 1 << 30, ea.FA_ERR_MISALIGNED),
])
def test_split_host_checks(lib, splits, ws, nbytes, want):
    rc = ea.fa_fwd_split(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 128, 0.1, 0, 0, splits,
                         ws, nbytes, (1.0, 1.0, 1.0), None, None)
    assert rc == want


@pytest.mark.parametrize("blk,want", [
    ((0, FAKE, FAKE), ea.FA_ERR_INVALID_ARG),
    ((FAKE, FAKE, 0), ea.FA_ERR_INVALID_ARG),
    ((FAKE, FAKE + 2, FAKE), ea.FA_ERR_MISALIGNED),
])
def test_blockscaled_host_checks(lib, blk, want):
    rc = ea.fa_fwd_fp8_blockscaled(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 128, 0.1, 0, *blk)
    assert rc == want


def test_blockscaled_shares_the_shape_checks(lib):
    assert ea.fa_fwd_fp8_blockscaled(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 96, 0.1, 0, FAKE,
                                     FAKE, FAKE) == ea.FA_ERR_UNSUPPORTED
    assert ea.fa_fwd_fp8_blockscaled(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 128, 0.1, 0, FAKE,
                                     FAKE, FAKE, 2, 0, 0) == ea.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("args,want", [
    ((0, FAKE, FAKE, 1, 1, 128, 128, None), ea.FA_ERR_INVALID_ARG),
    ((FAKE, FAKE, 0, 1, 1, 128, 128, None), ea.FA_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, 1, 0, 128, 128, None), ea.FA_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, 1, 1, 128, 32, None), ea.FA_ERR_UNSUPPORTED),
    ((FAKE, FAKE, FAKE, 256, 256, 128, 128, None), ea.FA_ERR_UNSUPPORTED),
    ((FAKE + 8, FAKE, FAKE, 1, 1, 128, 128, None), ea.FA_ERR_MISALIGNED),
    ((FAKE, FAKE, FAKE + 1, 1, 1, 128, 128, None), ea.FA_ERR_MISALIGNED),
    ((FAKE, FAKE, FAKE, 1, 1, 128, 128, FAKE + 4), ea.FA_ERR_MISALIGNED),
])
def test_quantize_host_checks(lib, args, want):
    assert ea.fa_quantize_e4m3(*args, 0, None) == want


def test_quantize_rejects_unknown_flags(lib):
    assert ea.fa_quantize_e4m3(FAKE, FAKE, FAKE, 1, 1, 128, 128, None, 2, None) == \
        ea.FA_ERR_INVALID_ARG


def test_bwd_workspace_bytes(lib):
    assert ea.bwd_workspace_bytes(1, 2, 300) == (2 * 300 * 4 + 255) // 256 * 256
    assert ea.bwd_workspace_bytes(0, 1, 8) == 0


@pytest.mark.parametrize("patch,want", [
    ({0: 0}, ea.FA_ERR_INVALID_ARG),            # null q
    ({15: 0}, ea.FA_ERR_INVALID_ARG),           # null workspace
    ({16: 16}, ea.FA_ERR_INVALID_ARG),          # workspace too small
    ({12: 96}, ea.FA_ERR_UNSUPPORTED),          # d = 96
    ({13: -1.0}, ea.FA_ERR_INVALID_ARG),        # negative scale
    ({6: FAKE + 8}, ea.FA_ERR_MISALIGNED),      # dq misaligned
    ({4: FAKE + 2}, ea.FA_ERR_MISALIGNED),      # lse misaligned
])
def test_bwd_host_checks(lib, patch, want):
    args = [FAKE] * 9 + [1, 1, 128, 128, 0.1, 0, FAKE, ea.bwd_workspace_bytes(1, 1, 128), None,
                         None]
    for i, val in patch.items():
        args[i] = val
    assert ea.fa_bwd(*args) == want
