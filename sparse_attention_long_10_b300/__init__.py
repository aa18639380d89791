"""Python binding of libnsa.so (include/nsa.h): argument marshalling only.

Every step of the NSA / DSA hot path runs in the library's CUDA kernels.  The
functions here take torch tensors (device memory, owned by the caller), pass
their raw pointers and the current CUDA stream through ctypes, and raise
``NsaError`` on a non-zero status.  There is no CPU fallback: the first use of
the library (any call, or the ``lib`` attribute) raises ImportError if
libnsa.so has not been built (``python -m sparse_attention_long_10_b300.build``).
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

import torch

__all__ = [
    "NsaError", "NsaCfg", "DsaCfg", "LIB_PATH", "lib", "make_cfg", "make_dsa_cfg",
    "NSA_LAYOUT_BTGD", "NSA_LAYOUT_BGTD", "NSA_FLAG_KC_GIVEN", "NSA_FLAG_TEST_STALL",
    "nsa_status_string", "nsa_version", "nsa_num_compressed",
    "nsa_compress_workspace_size", "nsa_prefill_workspace_size", "nsa_decode_workspace_size",
    "dsa_decode_workspace_size", "nsa_compress_kv", "nsa_compress_kv_noalloc",
    "nsa_compress_kv_noalloc_status", "nsa_full_attn_workspace_size", "nsa_full_attn_fwd",
    "nsa_decode_multi_workspace_size", "nsa_decode_multi", "nsa_prefill_fwd",
    "nsa_prefill_bwd_workspace_size", "nsa_prefill_bwd", "nsa_prefill_fwd_train", "nsa_decode_step",
    "dsa_decode_step", "nsa_device_status", "nsa_profile_enable", "nsa_profile_read", "workspace",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libnsa.so")

NSA_LAYOUT_BTGD = 0
NSA_LAYOUT_BGTD = 1
NSA_FLAG_KC_GIVEN = 1
NSA_FLAG_TEST_STALL = 0x80000000

_c_int, _c_float, _c_uint, _c_vp, _c_size = (ctypes.c_int, ctypes.c_float, ctypes.c_uint,
                                             ctypes.c_void_p, ctypes.c_size_t)


class NsaCfg(ctypes.Structure):
    """Mirror of ``nsa_cfg`` (include/nsa.h)."""
    _fields_ = [("B", _c_int), ("T", _c_int), ("H", _c_int), ("G", _c_int), ("dk", _c_int),
                ("dv", _c_int), ("l", _c_int), ("d", _c_int), ("lsel", _c_int), ("n", _c_int),
                ("w", _c_int), ("scale", _c_float), ("flags", _c_uint), ("pe_k", _c_vp),
                ("pe_v", _c_vp), ("w_k", _c_vp), ("w_v", _c_vp)]


class DsaCfg(ctypes.Structure):
    """Mirror of ``dsa_cfg`` (include/nsa.h)."""
    _fields_ = [("B", _c_int), ("T", _c_int), ("HI", _c_int), ("dI", _c_int), ("H", _c_int),
                ("dk", _c_int), ("dv", _c_int), ("topk", _c_int), ("scale", _c_float)]


class NsaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {nsa_status_string(code)} ({code})")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libnsa.so is not built ({LIB_PATH}); run "
                          "`python -m sparse_attention_long_10_b300.build`")
    L = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER
    sig = {
        "nsa_status_string": (ctypes.c_char_p, [_c_int]),
        "nsa_version": (_c_int, []),
        "nsa_num_compressed": (_c_int, [P(NsaCfg)]),
        "nsa_compress_workspace_size": (_c_size, [P(NsaCfg)]),
        "nsa_prefill_workspace_size": (_c_size, [P(NsaCfg)]),
        "nsa_decode_workspace_size": (_c_size, [P(NsaCfg)]),
        "dsa_decode_workspace_size": (_c_size, [P(DsaCfg)]),
        "dsa_prefill_workspace_size": (_c_size, [P(DsaCfg)]),
        "dsa_prefill_fwd": (_c_int, [P(DsaCfg), _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp,
                                     _c_vp, _c_size, _c_vp]),
        "nsa_compress_kv": (_c_int, [P(NsaCfg), _c_int, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_size,
                                     _c_vp]),
        "nsa_prefill_fwd": (_c_int, [P(NsaCfg), _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp,
                                     _c_vp, _c_vp, _c_size, _c_vp]),
        "nsa_decode_step": (_c_int, [P(NsaCfg), _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp,
                                     _c_vp, _c_vp, _c_size, _c_vp]),
        "dsa_decode_step": (_c_int, [P(DsaCfg), _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp,
                                     _c_vp, _c_vp, _c_vp, _c_size, _c_vp]),
        "nsa_device_status": (_c_int, [_c_vp, _c_vp]),
        "nsa_full_attn_workspace_size": (_c_size, [P(NsaCfg)]),
        "nsa_prefill_bwd_workspace_size": (_c_size, [P(NsaCfg)]),
        "nsa_prefill_bwd": (_c_int, [P(NsaCfg)] + [_c_vp] * 18 + [_c_vp, _c_size, _c_vp]),
        "nsa_prefill_fwd_train": (_c_int, [P(NsaCfg)] + [_c_vp] * 10 + [_c_vp, _c_size, _c_vp]),
        "nsa_decode_multi_workspace_size": (_c_size, [P(NsaCfg), _c_int]),
        "nsa_decode_multi": (_c_int, [P(NsaCfg), _c_int, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp,
                                      _c_vp, _c_size, _c_vp]),
        "nsa_full_attn_fwd": (_c_int, [P(NsaCfg), _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_size, _c_vp]),
        "nsa_compress_kv_noalloc": (_c_int, [P(NsaCfg), _c_int, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp]),
        "nsa_compress_kv_noalloc_status": (_c_int, [_c_vp]),
        "nsa_profile_enable": (_c_int, [_c_int]),
        "nsa_profile_read": (_c_int, [_c_int, ctypes.c_char_p, _c_size, ctypes.POINTER(_c_int),
                                      ctypes.POINTER(_c_float)]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name, None)
        if f is None:
            continue
        f.restype = res
        f.argtypes = args
    return L


_LIB = None


def _lib() -> ctypes.CDLL:
    global _LIB
    if _LIB is None:
        _LIB = _load()
    return _LIB


def __getattr__(name):
    if name == "lib":
        return _lib()
    raise AttributeError(name)


# ------------------------------------------------------------------ helpers
def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError("tensors passed to libnsa must be contiguous")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int, where: str):
    if rc != 0:
        raise NsaError(rc, where)


def make_cfg(B, T, H, G, dk, dv, phi=None, l=32, d=16, lsel=64, n=16, w=512, scale=0.0,
             flags=0) -> NsaCfg:
    """Build an ``nsa_cfg``.  ``phi`` = dict(pe_k, pe_v, w_k, w_v) of device tensors."""
    c = NsaCfg(B, T, H, G, dk, dv, l, d, lsel, n, w, float(scale), flags, None, None, None, None)
    if phi is not None:
        c.pe_k, c.pe_v = _ptr(phi["pe_k"]), _ptr(phi["pe_v"])
        c.w_k, c.w_v = _ptr(phi["w_k"]), _ptr(phi["w_v"])
    return c


def make_dsa_cfg(B, T, HI, dI, H, dk, dv, topk, scale=0.0) -> DsaCfg:
    return DsaCfg(B, T, HI, dI, H, dk, dv, topk, float(scale))


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """Caller-owned workspace (uint8, 256-byte aligned by the caching allocator)."""
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


# ------------------------------------------------------------------ ABI wrappers
def nsa_status_string(code: int) -> str:
    return _lib().nsa_status_string(code).decode()


def nsa_version() -> int:
    return _lib().nsa_version()


def nsa_num_compressed(cfg: NsaCfg) -> int:
    return _lib().nsa_num_compressed(ctypes.byref(cfg))


def nsa_compress_workspace_size(cfg: NsaCfg) -> int:
    return _lib().nsa_compress_workspace_size(ctypes.byref(cfg))


def nsa_prefill_workspace_size(cfg: NsaCfg) -> int:
    return _lib().nsa_prefill_workspace_size(ctypes.byref(cfg))


def nsa_decode_workspace_size(cfg: NsaCfg) -> int:
    return _lib().nsa_decode_workspace_size(ctypes.byref(cfg))


def dsa_decode_workspace_size(cfg: DsaCfg) -> int:
    return _lib().dsa_decode_workspace_size(ctypes.byref(cfg))


def nsa_compress_kv(cfg: NsaCfg, layout: int, k, v, kc, vc, ws, stream=None):
    _check(_lib().nsa_compress_kv(ctypes.byref(cfg), layout, _ptr(k), _ptr(v), _ptr(kc), _ptr(vc),
                               _ptr(ws), ws.numel() if ws is not None else 0, _stream(stream)),
           "nsa_compress_kv")


def nsa_compress_kv_noalloc(cfg: NsaCfg, layout: int, k, v, kc, vc, stream=None):
    """Compression with the library's fixed scratch array: no workspace and no
    allocation, for callers that cannot allocate device memory."""
    _check(_lib().nsa_compress_kv_noalloc(ctypes.byref(cfg), layout, _ptr(k), _ptr(v), _ptr(kc), _ptr(vc),
                                       _stream(stream)), "nsa_compress_kv_noalloc")


def nsa_compress_kv_noalloc_status(stream=None) -> int:
    """Status word of the no-alloc call's fixed array (synchronises, clears)."""
    return _lib().nsa_compress_kv_noalloc_status(_stream(stream))


def nsa_prefill_fwd(cfg: NsaCfg, q, k, v, gates, kc, vc, out, idx_out, ws, stream=None):
    _check(_lib().nsa_prefill_fwd(ctypes.byref(cfg), _ptr(q), _ptr(k), _ptr(v), _ptr(gates),
                               _ptr(kc), _ptr(vc), _ptr(out), _ptr(idx_out), _ptr(ws),
                               ws.numel() if ws is not None else 0, _stream(stream)),
           "nsa_prefill_fwd")


def nsa_prefill_bwd_workspace_size(cfg: NsaCfg) -> int:
    return int(_lib().nsa_prefill_bwd_workspace_size(ctypes.byref(cfg)))


def nsa_prefill_fwd_train(cfg: NsaCfg, q, k, v, gates, kc, vc, out, idx_out, slc_lse, slc_o, ws, stream=None):
    _check(_lib().nsa_prefill_fwd_train(ctypes.byref(cfg), _ptr(q), _ptr(k), _ptr(v), _ptr(gates), _ptr(kc),
                                        _ptr(vc), _ptr(out), _ptr(idx_out), _ptr(slc_lse), _ptr(slc_o), _ptr(ws),
                                        ws.numel() if ws is not None else 0, _stream(stream)),
           "nsa_prefill_fwd_train")


def nsa_prefill_bwd(cfg: NsaCfg, q, k, v, gates, kc, vc, idx, dout, dq, dk, dv, dgates, dw_k, dw_v,
                    dpe_k, dpe_v, ws, stream=None, slc_lse=None, slc_o=None):
    """Gradients of sum(dout * out) for the forward on the same inputs; the
    outputs are fp32 tensors (see include/nsa.h).  slc_lse / slc_o: the
    statistics nsa_prefill_fwd_train saved (optional)."""
    _check(_lib().nsa_prefill_bwd(ctypes.byref(cfg), _ptr(q), _ptr(k), _ptr(v), _ptr(gates), _ptr(kc),
                                  _ptr(vc), _ptr(idx), _ptr(slc_lse), _ptr(slc_o), _ptr(dout), _ptr(dq),
                                  _ptr(dk), _ptr(dv), _ptr(dgates),
                                  _ptr(dw_k), _ptr(dw_v), _ptr(dpe_k), _ptr(dpe_v), _ptr(ws),
                                  ws.numel() if ws is not None else 0, _stream(stream)),
           "nsa_prefill_bwd")


def nsa_full_attn_workspace_size(cfg: NsaCfg) -> int:
    return _lib().nsa_full_attn_workspace_size(ctypes.byref(cfg))


def nsa_full_attn_fwd(cfg: NsaCfg, q, k, v, out, ws, stream=None):
    """Exact causal full attention (the dense comparison)."""
    _check(_lib().nsa_full_attn_fwd(ctypes.byref(cfg), _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(ws),
                                 ws.numel() if ws is not None else 0, _stream(stream)), "nsa_full_attn_fwd")


def nsa_decode_multi_workspace_size(cfg: NsaCfg, m: int) -> int:
    return _lib().nsa_decode_multi_workspace_size(ctypes.byref(cfg), m)


def nsa_decode_multi(cfg: NsaCfg, m: int, q, kcache, vcache, kc, vc, gates, out, idx_out, ws, stream=None):
    """m new tokens per sequence (rows T-m .. T-1) from head-major caches."""
    _check(_lib().nsa_decode_multi(ctypes.byref(cfg), m, _ptr(q), _ptr(kcache), _ptr(vcache), _ptr(kc), _ptr(vc),
                                _ptr(gates), _ptr(out), _ptr(idx_out), _ptr(ws),
                                ws.numel() if ws is not None else 0, _stream(stream)), "nsa_decode_multi")


def nsa_decode_step(cfg: NsaCfg, q, kcache, vcache, kc, vc, gates, out, idx_out, ws, stream=None,
                    seq_lens=None):
    """seq_lens: optional int32 device tensor [B] of sequence lengths (None: all cfg.T)."""
    _check(_lib().nsa_decode_step(ctypes.byref(cfg), _ptr(q), _ptr(kcache), _ptr(vcache), _ptr(kc),
                               _ptr(vc), _ptr(seq_lens), _ptr(gates), _ptr(out), _ptr(idx_out), _ptr(ws),
                               ws.numel() if ws is not None else 0, _stream(stream)),
           "nsa_decode_step")


def dsa_decode_step(cfg: DsaCfg, qI, wI, kI, q, k, v, out, idx_out, ws, stream=None, seq_lens=None):
    """seq_lens: optional int32 device tensor [B] of context lengths (None: all cfg.T)."""
    _check(_lib().dsa_decode_step(ctypes.byref(cfg), _ptr(qI), _ptr(wI), _ptr(kI), _ptr(q), _ptr(k),
                               _ptr(v), _ptr(seq_lens), _ptr(out), _ptr(idx_out), _ptr(ws),
                               ws.numel() if ws is not None else 0, _stream(stream)),
           "dsa_decode_step")


def dsa_prefill_workspace_size(cfg: DsaCfg) -> int:
    return _lib().dsa_prefill_workspace_size(ctypes.byref(cfg))


def dsa_prefill_fwd(cfg: DsaCfg, qI, wI, kI, q, k, v, out, idx_out, ws, stream=None):
    """Every position of every sequence a query; v None: latent values."""
    _check(_lib().dsa_prefill_fwd(ctypes.byref(cfg), _ptr(qI), _ptr(wI), _ptr(kI), _ptr(q), _ptr(k),
                               _ptr(v), _ptr(out), _ptr(idx_out), _ptr(ws),
                               ws.numel() if ws is not None else 0, _stream(stream)),
           "dsa_prefill_fwd")


def nsa_device_status(ws, stream=None) -> int:
    return _lib().nsa_device_status(_ptr(ws), _stream(stream))


def nsa_profile_enable(on: bool = True) -> None:
    _lib().nsa_profile_enable(1 if on else 0)


def nsa_profile_read(max_kernels: int = 32):
    """{kernel name: (launches, total device ms)} since the last read."""
    names = ctypes.create_string_buffer(4096)
    cnt = (_c_int * max_kernels)()
    tot = (_c_float * max_kernels)()
    n = _lib().nsa_profile_read(max_kernels, names, 4096, cnt, tot)
    if n < 0:
        raise NsaError(-n, "nsa_profile_read")
    keys = names.value.decode().split(",") if n else []
    return {k: (cnt[i], tot[i]) for i, k in enumerate(keys)}
