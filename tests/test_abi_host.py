"""C-ABI host tests (CPU): the library builds, loads, exports every entry point
that include/nsa.h declares, and rejects bad arguments with the documented
status codes before any CUDA work."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def nsa():
    from sparse_attention_long_10_b300 import build
    build.build()
    import sparse_attention_long_10_b300 as m
    return m


def _declared_functions():
    hdr = open(os.path.join(ROOT, "include", "nsa.h")).read()
    hdr = re.sub(r"/\*.*?\*/", "", hdr, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*((?:nsa|dsa)_\w+)\s*\(", hdr, flags=re.M)
    return sorted(set(names))


def test_header_declares_entry_points():
    names = _declared_functions()
    for must in ("nsa_compress_kv", "nsa_prefill_fwd", "nsa_decode_step", "dsa_decode_step",
                 "nsa_status_string", "nsa_device_status"):
        assert must in names


def test_library_exports_every_declared_symbol(nsa):
    lib = ctypes.CDLL(nsa.LIB_PATH)
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(nsa):
    assert nsa.nsa_status_string(0) == "NSA_OK"
    assert nsa.nsa_status_string(4) == "NSA_ERR_WORKSPACE"
    assert nsa.nsa_status_string(999) == "NSA_ERR_UNKNOWN"
    assert nsa.nsa_version() >= 100


def test_cfg_struct_layout(nsa):
    # 11 ints, float, unsigned, then 4 pointers aligned to 8
    assert ctypes.sizeof(nsa.NsaCfg) == 56 + 32
    assert nsa.NsaCfg.pe_k.offset == 56
    assert ctypes.sizeof(nsa.DsaCfg) == 36


def test_num_compressed_and_workspace(nsa):
    c = nsa.make_cfg(1, 65536, 64, 4, 192, 128)
    assert nsa.nsa_num_compressed(c) == 4095
    assert nsa.nsa_compress_workspace_size(c) > 0
    bad = nsa.make_cfg(1, 65536, 64, 3, 192, 128)     # H % G != 0
    assert nsa.nsa_num_compressed(bad) == -1
    assert nsa.nsa_compress_workspace_size(bad) == 0


FAKE = 1 << 20            # a 16-byte aligned non-null "device" address; never dereferenced


@pytest.mark.parametrize("mutate,code", [
    (dict(H=64, G=3), 1),            # H % G
    (dict(B=0), 1),                  # non-positive
    (dict(dk=100), 2),               # dk not a multiple of 64
    (dict(l=64), 2),                 # only l=32 is implemented
    (dict(H=48, G=1), 2),            # heads per group not a power of two
    (dict(n=2), 2),                  # fewer than the 3 forced blocks
])
def test_compress_rejects_bad_cfg(nsa, mutate, code):
    base = dict(B=1, T=4096, H=64, G=4, dk=192, dv=128)
    base.update(mutate)
    c = nsa.make_cfg(**base)
    c.pe_k = c.pe_v = c.w_k = c.w_v = FAKE
    rc = nsa.lib.nsa_compress_kv(ctypes.byref(c), 0, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 20, None)
    assert rc == code


def test_compress_rejects_pointers_and_workspace(nsa):
    c = nsa.make_cfg(1, 4096, 64, 4, 192, 128)
    c.pe_k = c.pe_v = c.w_k = c.w_v = FAKE
    ws_need = nsa.nsa_compress_workspace_size(c)
    f = nsa.lib.nsa_compress_kv
    assert f(None, 0, FAKE, FAKE, FAKE, FAKE, FAKE, ws_need, None) == 1
    assert f(ctypes.byref(c), 7, FAKE, FAKE, FAKE, FAKE, FAKE, ws_need, None) == 1      # layout
    assert f(ctypes.byref(c), 0, None, FAKE, FAKE, FAKE, FAKE, ws_need, None) == 1
    assert f(ctypes.byref(c), 0, FAKE + 2, FAKE, FAKE, FAKE, FAKE, ws_need, None) == 3  # misaligned
    assert f(ctypes.byref(c), 0, FAKE, FAKE, FAKE, FAKE, FAKE + 16, ws_need, None) == 3  # ws 256-aligned
    assert f(ctypes.byref(c), 0, FAKE, FAKE, FAKE, FAKE, FAKE, ws_need - 1, None) == 4
    c.w_v = None
    assert f(ctypes.byref(c), 0, FAKE, FAKE, FAKE, FAKE, FAKE, ws_need, None) == 1


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_valid_call_without_device_reports_no_device(nsa):
    c = nsa.make_cfg(1, 4096, 64, 4, 192, 128)
    c.pe_k = c.pe_v = c.w_k = c.w_v = FAKE
    rc = nsa.lib.nsa_compress_kv(ctypes.byref(c), 0, FAKE, FAKE, FAKE, FAKE, FAKE,
                                 nsa.nsa_compress_workspace_size(c), None)
    assert rc == 7


def test_dsa_latent_values_argument_checks(nsa):
    """dsa_decode_step with v == NULL reads the values from the key rows; that
    needs dv <= dk (else INVALID_ARG), and a given v must be 16-byte aligned."""
    f = nsa.lib.dsa_decode_step
    c = nsa.make_dsa_cfg(8, 131072, 4, 64, 16, 576, 512, 2048)
    need = nsa.dsa_decode_workspace_size(c)
    assert need > 0
    bad = nsa.make_dsa_cfg(8, 131072, 4, 64, 16, 64, 128, 2048)   # dv > dk
    assert f(ctypes.byref(bad), FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, None, FAKE,
             nsa.dsa_decode_workspace_size(bad), None) == 1
    assert f(ctypes.byref(c), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE + 2, FAKE, None, FAKE, need, None) == 3
    if not torch.cuda.is_available():
        # valid arguments, latent or not: the no-device status
        assert f(ctypes.byref(c), FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, None, FAKE, need, None) == 7
        assert f(ctypes.byref(c), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, need, None) == 7
