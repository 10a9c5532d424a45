"""Host-side checks of the C ABI (no GPU work): the library loads, exports every function
include/sdcp.h declares, and rejects bad arguments before any launch."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "sdcp.h")


@pytest.fixture(scope="module")
def libsdcp():
    from speculative_decoding_verification_sdcp_gb300 import build_ext
    path = build_ext.build()
    return ctypes.CDLL(path)


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s+\**\s*(sdcp_[a-z0-9_]+)\s*\(",
                       src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("sdcp_verify_batch", "sdcp_workspace_bytes", "sdcp_row_stats", "sdcp_strerror",
              "sdcp_abi_version"):
        assert n in names


def test_every_declared_symbol_is_exported(libsdcp):
    for n in declared_functions():
        assert hasattr(libsdcp, n), n


def test_host_only_calls(libsdcp):
    libsdcp.sdcp_strerror.restype = ctypes.c_char_p
    libsdcp.sdcp_workspace_bytes.restype = ctypes.c_size_t
    libsdcp.sdcp_workspace_bytes.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int64]
    assert libsdcp.sdcp_abi_version() == 2
    assert b"success" in libsdcp.sdcp_strerror(0)
    assert libsdcp.sdcp_workspace_bytes(32000, 64, 512) >= (2 * 512 + 64) * 32
    assert libsdcp.sdcp_workspace_bytes(0, 64, 512) == 0
    assert libsdcp.sdcp_workspace_bytes(100, -1, 0) == 0
    assert libsdcp.sdcp_workspace_bytes((1 << 24) + 1, 1, 1) == 0


def test_argument_errors_before_launch(libsdcp):
    f = libsdcp.sdcp_verify_batch
    vp = ctypes.c_void_p
    f.argtypes = [vp, vp, ctypes.c_int, ctypes.c_int64, ctypes.c_int32, vp, ctypes.c_int64, vp, vp,
                  vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
    f.restype = ctypes.c_int
    fake = vp(4096)
    # B = 0: nothing to do, success without touching the device
    assert f(None, None, 0, 10, 0, None, 0, None, None, None, None, None, None, None, 0, None) == 0
    # negative B, V < 1, bad dtype, null pointers
    assert f(fake, fake, 0, 10, -1, fake, 0, fake, fake, fake, fake, fake, fake, fake, 1 << 20, None) == 1
    assert f(fake, fake, 0, 0, 1, fake, 0, fake, fake, fake, fake, fake, fake, fake, 1 << 20, None) == 1
    assert f(fake, fake, 7, 10, 1, fake, 0, fake, fake, fake, fake, fake, fake, fake, 1 << 20, None) == 1
    assert f(None, fake, 0, 10, 1, fake, 0, fake, fake, fake, fake, fake, fake, fake, 1 << 20, None) == 1
    # misaligned logits pointer (f32 needs 4-byte alignment)
    assert f(vp(4097), fake, 0, 10, 1, fake, 1, fake, fake, fake, fake, fake, fake, fake, 1 << 20, None) == 3
    # workspace too small or misaligned
    assert f(fake, fake, 0, 10, 1, fake, 1, fake, fake, fake, fake, fake, fake, fake, 16, None) == 2
    assert f(fake, fake, 0, 10, 1, fake, 1, fake, fake, fake, fake, fake, fake, vp(4100), 1 << 20, None) == 2
    # vocabulary above the maximum
    assert f(fake, fake, 0, (1 << 24) + 1, 1, fake, 1, fake, fake, fake, fake, fake, fake, fake, 1 << 20, None) == 4
