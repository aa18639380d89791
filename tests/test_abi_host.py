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
    assert f(ctypes.byref(bad), FAKE, FAKE, FAKE, FAKE, FAKE, None, None, FAKE, None, FAKE,
             nsa.dsa_decode_workspace_size(bad), None) == 1
    assert f(ctypes.byref(c), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE + 2, None, FAKE, None, FAKE, need, None) == 3
    # per-row context lengths: an int32 array, 4-byte aligned
    assert f(ctypes.byref(c), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE + 2, FAKE, None, FAKE, need, None) == 3
    if not torch.cuda.is_available():
        # valid arguments, latent or not, with or without lengths: the no-device status
        assert f(ctypes.byref(c), FAKE, FAKE, FAKE, FAKE, FAKE, None, None, FAKE, None, FAKE, need, None) == 7
        assert f(ctypes.byref(c), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, None, FAKE, need, None) == 7
        assert f(ctypes.byref(c), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE + 4, FAKE, None, FAKE, need, None) == 7


def test_dsa_prefill_argument_checks(nsa):
    """dsa_prefill_fwd: every position of every sequence is a query row, so
    B*T rows must fit the launch grid (<= 65535, else UNSUPPORTED); the
    pointer rules are those of dsa_decode_step."""
    f = nsa.lib.dsa_prefill_fwd
    c = nsa.make_dsa_cfg(1, 8192, 4, 64, 16, 576, 512, 2048)
    need = nsa.dsa_prefill_workspace_size(c)
    assert need > nsa.dsa_decode_workspace_size(nsa.make_dsa_cfg(1, 8192, 4, 64, 16, 576, 512, 2048))
    # B*T = 65,536 rows: unsupported, and no workspace size
    big = nsa.make_dsa_cfg(2, 32768, 4, 64, 16, 576, 512, 2048)
    assert nsa.dsa_prefill_workspace_size(big) == 0
    assert f(ctypes.byref(big), FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, None, FAKE, 1 << 40, None) == 2
    # latent values need dv <= dk; a given v must be 16-byte aligned
    bad = nsa.make_dsa_cfg(1, 4096, 4, 64, 16, 64, 128, 2048)
    assert f(ctypes.byref(bad), FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, None, FAKE,
             nsa.dsa_prefill_workspace_size(bad), None) == 1
    assert f(ctypes.byref(c), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE + 2, FAKE, None, FAKE, need, None) == 3
    # null inputs, misaligned idx_out, a short workspace
    assert f(ctypes.byref(c), None, FAKE, FAKE, FAKE, FAKE, None, FAKE, None, FAKE, need, None) == 1
    assert f(ctypes.byref(c), FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE + 4, FAKE, need, None) == 3
    assert f(ctypes.byref(c), FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, None, FAKE, need - 256, None) == 4
    if not torch.cuda.is_available():
        assert f(ctypes.byref(c), FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, None, FAKE, need, None) == 7
        assert f(ctypes.byref(c), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, need, None) == 7


def _prefill_args(nsa, c, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, gates=FAKE, kc=FAKE, vc=FAKE, out=FAKE, idx=None, ws=FAKE,
             ws_bytes=nsa.nsa_prefill_workspace_size(c))
    a.update(kw)
    return nsa.lib.nsa_prefill_fwd(ctypes.byref(c), a["q"], a["k"], a["v"], a["gates"], a["kc"], a["vc"],
                                   a["out"], a["idx"], a["ws"], a["ws_bytes"], None)


def test_prefill_argument_checks(nsa):
    c = nsa.make_cfg(1, 4096, 64, 4, 192, 128)
    c.pe_k = c.pe_v = c.w_k = c.w_v = FAKE
    need = nsa.nsa_prefill_workspace_size(c)
    # the workspace holds the fp32 cmp+win partial and the kept-block lists
    assert need >= 4096 * 64 * 128 * 4 + 4096 * 4 * 16 * 4        # fp32 partial + kept blocks
    assert nsa.nsa_prefill_workspace_size(nsa.make_cfg(1, 8192, 64, 4, 192, 128)) > need
    assert _prefill_args(nsa, c, q=None) == 1
    assert _prefill_args(nsa, c, k=FAKE + 2) == 3
    assert _prefill_args(nsa, c, idx=FAKE + 4) == 3
    assert _prefill_args(nsa, c, kc=None) == 1                     # a cache exists at T = 4096
    assert _prefill_args(nsa, c, ws=FAKE + 16) == 3
    assert _prefill_args(nsa, c, ws_bytes=need - 1) == 4
    c.w_k = None                                                   # phi needed to build the cache ...
    assert _prefill_args(nsa, c) == 1
    c.flags = nsa.NSA_FLAG_KC_GIVEN                                # ... but not when it is given
    if not torch.cuda.is_available():
        assert _prefill_args(nsa, c) == 7
        short = nsa.make_cfg(1, 20, 64, 4, 192, 128)               # T < l: no cache, kc/vc may be NULL
        short.pe_k = short.pe_v = short.w_k = short.w_v = FAKE
        assert _prefill_args(nsa, short, kc=None, vc=None,
                             ws_bytes=nsa.nsa_prefill_workspace_size(short)) == 7


@pytest.mark.parametrize("shape", [
    dict(H=64, G=2),       # 32 heads per group: the kernels take at most 16
    dict(T=70000),         # longer than the prefill kernels' 65,536
    dict(dv=192),          # prefill values are 64 or 128 wide
    dict(n=17),            # at most 16 kept blocks in prefill
])
def test_prefill_rejects_unimplemented_shapes(nsa, shape):
    base = dict(B=1, T=4096, H=64, G=4, dk=192, dv=128)
    n = shape.pop("n", 16)
    base.update(shape)
    c = nsa.make_cfg(**base, n=n)
    c.pe_k = c.pe_v = c.w_k = c.w_v = FAKE
    assert _prefill_args(nsa, c, ws_bytes=1 << 40) == 2


def test_decode_argument_checks(nsa):
    c = nsa.make_cfg(16, 65536, 64, 4, 192, 128)
    need = nsa.nsa_decode_workspace_size(c)
    assert need > 0
    f = nsa.lib.nsa_decode_step

    def call(**kw):
        a = dict(q=FAKE, kcache=FAKE, vcache=FAKE, kc=FAKE, vc=FAKE, gates=FAKE, out=FAKE, idx=None, ws=FAKE,
                 ws_bytes=need)
        a.update(kw)
        return f(ctypes.byref(c), a["q"], a["kcache"], a["vcache"], a["kc"], a["vc"], a.get("lens"), a["gates"],
                 a["out"], a["idx"], a["ws"], a["ws_bytes"], None)
    assert call(kcache=None) == 1
    assert call(gates=FAKE + 8) == 3
    assert call(vc=None) == 1
    assert call(ws_bytes=need - 1) == 4
    assert call(lens=FAKE + 2) == 3                                 # int32 lengths, 4-byte aligned
    if not torch.cuda.is_available():
        assert call() == 7
        assert call(lens=FAKE + 4) == 7                             # a device array of lengths
    wide = nsa.make_cfg(16, 65536, 64, 2, 192, 128)                # 32 heads per group
    assert nsa.nsa_decode_workspace_size(wide) == 0
    assert f(ctypes.byref(wide), FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, None, FAKE, 1 << 40, None) == 2


@pytest.mark.parametrize("mutate", [
    dict(H=64, G=3), dict(B=0), dict(dk=100), dict(l=64), dict(H=48, G=1), dict(n=2), dict(T=0),
    dict(dv=320),
])
def test_noalloc_rejects_bad_cfg_like_the_workspace_call(nsa, mutate):
    """The allocation-free compression applies the same argument rules as
    nsa_compress_kv and returns the same codes."""
    base = dict(B=1, T=4096, H=64, G=4, dk=192, dv=128)
    base.update(mutate)
    c = nsa.make_cfg(**base)
    c.pe_k = c.pe_v = c.w_k = c.w_v = FAKE
    rc_ws = nsa.lib.nsa_compress_kv(ctypes.byref(c), 0, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 30, None)
    rc_na = nsa.lib.nsa_compress_kv_noalloc(ctypes.byref(c), 0, FAKE, FAKE, FAKE, FAKE, None)
    assert rc_ws != 0 and rc_na == rc_ws


def test_noalloc_argument_checks_match(nsa):
    c = nsa.make_cfg(1, 4096, 64, 4, 192, 128)
    c.pe_k = c.pe_v = c.w_k = c.w_v = FAKE
    f_ws = lambda *p: nsa.lib.nsa_compress_kv(ctypes.byref(c), *p, FAKE, 1 << 30, None)
    f_na = lambda *p: nsa.lib.nsa_compress_kv_noalloc(ctypes.byref(c), *p, None)
    for args in [(7, FAKE, FAKE, FAKE, FAKE), (0, None, FAKE, FAKE, FAKE), (0, FAKE + 2, FAKE, FAKE, FAKE),
                 (0, FAKE, FAKE, None, FAKE), (0, FAKE, FAKE, FAKE, FAKE + 8)]:
        assert f_na(*args) == f_ws(*args) != 0
    assert nsa.lib.nsa_compress_kv_noalloc(None, 0, FAKE, FAKE, FAKE, FAKE, None) == 1
    c.pe_v = FAKE + 4
    assert f_na(0, FAKE, FAKE, FAKE, FAKE) == f_ws(0, FAKE, FAKE, FAKE, FAKE) == 3
    if not torch.cuda.is_available():
        c.pe_v = FAKE
        assert f_na(0, FAKE, FAKE, FAKE, FAKE) == 7
        assert nsa.lib.nsa_compress_kv_noalloc_status(None) == 7


def test_full_attention_argument_checks(nsa):
    c = nsa.make_cfg(1, 4096, 64, 4, 192, 128)
    need = nsa.nsa_full_attn_workspace_size(c)
    assert need == 256                                   # the status word only
    f = nsa.lib.nsa_full_attn_fwd
    assert f(ctypes.byref(c), None, FAKE, FAKE, FAKE, FAKE, need, None) == 1
    assert f(ctypes.byref(c), FAKE, FAKE + 2, FAKE, FAKE, FAKE, need, None) == 3
    assert f(ctypes.byref(c), FAKE, FAKE, FAKE, FAKE, FAKE, need - 1, None) == 4
    wide = nsa.make_cfg(1, 4096, 64, 2, 192, 128)        # 32 heads per group
    assert nsa.nsa_full_attn_workspace_size(wide) == 0
    assert f(ctypes.byref(wide), FAKE, FAKE, FAKE, FAKE, FAKE, need, None) == 2
    if not torch.cuda.is_available():
        assert f(ctypes.byref(c), FAKE, FAKE, FAKE, FAKE, FAKE, need, None) == 7


def test_decode_multi_argument_checks(nsa):
    c = nsa.make_cfg(16, 65536, 64, 4, 192, 128)
    need = nsa.nsa_decode_multi_workspace_size(c, 4)
    assert need >= 256 + 16 * 4 * 64 * 128 * 4
    assert nsa.nsa_decode_multi_workspace_size(c, 0) == 0
    assert nsa.nsa_decode_multi_workspace_size(c, 65537) == 0
    f = nsa.lib.nsa_decode_multi

    def call(m=4, **kw):
        a = dict(q=FAKE, kcache=FAKE, vcache=FAKE, kc=FAKE, vc=FAKE, gates=FAKE, out=FAKE, idx=None, ws=FAKE,
                 ws_bytes=need)
        a.update(kw)
        return f(ctypes.byref(c), m, a["q"], a["kcache"], a["vcache"], a["kc"], a["vc"], a["gates"], a["out"],
                 a["idx"], a["ws"], a["ws_bytes"], None)
    assert call(m=0) == 1
    assert call(m=65537) == 1
    assert call(q=None) == 1
    assert call(vc=None) == 1
    assert call(out=FAKE + 2) == 3
    assert call(ws_bytes=need - 1) == 4
    if not torch.cuda.is_available():
        assert call() == 7


def test_prefill_backward_argument_checks(nsa):
    c = nsa.make_cfg(1, 65536, 64, 4, 192, 128)
    c.pe_k = c.pe_v = c.w_k = c.w_v = FAKE
    need = nsa.nsa_prefill_bwd_workspace_size(c)
    # the per-branch log-sum-exp and dg rows alone: 2 x 3 x T x H fp32
    assert need >= 256 + 2 * 3 * 65536 * 64 * 4
    f = nsa.lib.nsa_prefill_bwd

    def call(cfg=c, **kw):
        names = ["q", "k", "v", "gates", "kc", "vc", "idx", "slc_lse", "slc_o", "dout", "dq", "dk", "dv", "dgates",
                 "dw_k", "dw_v", "dpe_k", "dpe_v"]
        a = {n: FAKE for n in names}
        a.update(ws=FAKE, ws_bytes=need)
        a.update(kw)
        return f(ctypes.byref(cfg), *[a[n] for n in names], a["ws"], a["ws_bytes"], None)
    assert call(q=None) == 1
    assert call(idx=None) == 1
    assert call(dpe_v=None) == 1
    assert call(dout=FAKE + 2) == 3
    assert call(slc_o=None) == 1                         # the saved statistics come as a pair
    assert call(slc_lse=FAKE + 4) == 3
    assert call(ws=FAKE + 16) == 3                      # workspace must be 256-byte aligned
    assert call(ws_bytes=need - 1) == 4
    wide = nsa.make_cfg(1, 4096, 64, 2, 192, 128)       # 32 heads per group
    wide.pe_k = wide.pe_v = wide.w_k = wide.w_v = FAKE
    assert nsa.nsa_prefill_bwd_workspace_size(wide) == 0
    assert call(cfg=wide) == 2
    small_dk = nsa.make_cfg(1, 4096, 64, 4, 64, 128)    # dk 64 is not implemented by the backward
    small_dk.pe_k = small_dk.pe_v = small_dk.w_k = small_dk.w_v = FAKE
    assert call(cfg=small_dk) == 2
    c.w_v = None
    assert call() == 1
    c.w_v = FAKE
    if not torch.cuda.is_available():
        assert call() == 7


def test_prefill_fwd_train_argument_checks(nsa):
    c = nsa.make_cfg(1, 4096, 64, 4, 192, 128)
    c.pe_k = c.pe_v = c.w_k = c.w_v = FAKE
    need = nsa.nsa_prefill_workspace_size(c)
    f = nsa.lib.nsa_prefill_fwd_train

    def call(**kw):
        names = ["q", "k", "v", "gates", "kc", "vc", "out", "idx", "slc_lse", "slc_o"]
        a = {n: FAKE for n in names}
        a.update(ws=FAKE, ws_bytes=need)
        a.update(kw)
        return f(ctypes.byref(c), *[a[n] for n in names], a["ws"], a["ws_bytes"], None)
    assert call(idx=None) == 1                           # the kept blocks are required here
    assert call(slc_lse=None) == 1
    assert call(slc_o=FAKE + 8) == 3
    assert call(ws_bytes=need - 1) == 4
    if not torch.cuda.is_available():
        assert call() == 7
