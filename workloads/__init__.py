"""Seeded synthetic inputs for the NSA / DSA hot path.

This module is shared by the oracle (``oracle/``), the tests, ``bench.py`` and
``__graft_entry__.smoke``.  It holds NO arithmetic of the method itself: it
only draws random numbers, scales them and rounds them to bf16, so that the
oracle and the CUDA path read identical bytes.

Recipe (every workload): ``torch.Generator('cpu').manual_seed(seed)``; each
tensor is one ``torch.randn`` call in fp32, in the fixed order listed in each
generator, multiplied by its standard deviation and rounded to bf16 (round to
nearest even).  Gates are ``bf16(sigmoid(logits))`` with logits ~ N(0, 1).

Distributions (NSA pages, "Native Sparse Attention" overview, section II:
l=32, d=16, l'=64, n=16, w=512):
  Q, K, V           ~ N(0, 1)
  PE_K [l, dk], PE_V [l, dv]   ~ N(0, 0.02^2)      (0.02 is a std)
  W_cK [l*dk, dk]   ~ N(0, 1/(l*dk))               (1/(l*dk) is a variance)
  W_cV [l*dv, dv]   ~ N(0, 1/(l*dv))
DSA (page "DeepSeek Sparse Attention (DSA) principle"): every tensor ~ N(0,1).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import torch

__all__ = [
    "NSAParams", "PrefillWorkload", "DecodeWorkload", "DSAWorkload",
    "prefill_config", "decode_config", "dsa_config", "dsa_prefill_config",
    "make_prefill", "make_prefill_dout", "make_decode", "make_decode_multi", "make_dsa",
    "make_dsa_prefill", "PREFILL_CONFIGS",
]


@dataclasses.dataclass(frozen=True)
class NSAParams:
    """Branch hyper-parameters named on the NSA overview page (section II)."""
    l: int = 32        # compression block length
    d: int = 16        # compression stride
    lsel: int = 64     # selection block length l'
    n: int = 16        # selected blocks per query (block 0 + 2 local included)
    w: int = 512       # sliding-window length


@dataclasses.dataclass(frozen=True)
class PrefillWorkload:
    name: str
    B: int
    T: int
    H: int
    G: int
    dk: int
    dv: int
    seed: int
    params: NSAParams = NSAParams()


@dataclasses.dataclass(frozen=True)
class DecodeWorkload:
    name: str
    B: int
    T: int
    H: int
    G: int
    dk: int
    dv: int
    seed: int
    params: NSAParams = NSAParams()


@dataclasses.dataclass(frozen=True)
class DSAWorkload:
    name: str
    B: int
    T: int
    HI: int      # indexer heads
    dI: int      # indexer head dim
    H: int       # attention query heads
    dk: int
    dv: int
    topk: int
    seed: int


PREFILL_CONFIGS: Dict[str, PrefillWorkload] = {
    "tiny_2k": PrefillWorkload("nsa_prefill_T2048_H4_G1_d64", 1, 2048, 4, 1, 64, 64, 0),
    "prefill_8k": PrefillWorkload("nsa_prefill_T8192_H64_G4_dk192_dv128", 1, 8192, 64, 4, 192, 128, 1),
    "prefill_64k": PrefillWorkload("nsa_prefill_T65536_H64_G4_dk192_dv128", 1, 65536, 64, 4, 192, 128, 2),
}


def prefill_config(key: str) -> PrefillWorkload:
    return PREFILL_CONFIGS[key]


def decode_config() -> DecodeWorkload:
    """16 sequences x 65,536-token cache, 64 query heads / 4 KV heads."""
    return DecodeWorkload("nsa_decode_B16_T65536_H64_G4_dk192_dv128", 16, 65536, 64, 4, 192, 128, 3)


def dsa_config() -> DSAWorkload:
    """Batch 8, context 131,072, indexer 4x64, 16 heads, dk=576, dv=512, top-2048."""
    return DSAWorkload("dsa_decode_B8_T131072_HI4_dI64_H16_dk576_dv512_top2048",
                       8, 131072, 4, 64, 16, 576, 512, 2048, 4)


def dsa_prefill_config() -> DSAWorkload:
    """DSA prefill: one 8,192-token sequence, every position a query; indexer
    4x64, 16 heads, latent keys of 576 columns whose first 512 are the values,
    top-2048 (the decode step's heads and selection over a whole sequence)."""
    return DSAWorkload("dsa_prefill_B1_T8192_HI4_dI64_H16_dk576_dv512_top2048_latent",
                       1, 8192, 4, 64, 16, 576, 512, 2048, 13)


def _draw(gen: torch.Generator, shape, std: float) -> torch.Tensor:
    x = torch.randn(*shape, generator=gen, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def _gates(gen: torch.Generator, shape) -> torch.Tensor:
    logits = torch.randn(*shape, generator=gen, dtype=torch.float32)
    return torch.sigmoid(logits).to(torch.bfloat16)


def _phi_params(gen: torch.Generator, l: int, dk: int, dv: int):
    pe_k = _draw(gen, (l, dk), 0.02)
    pe_v = _draw(gen, (l, dv), 0.02)
    w_k = _draw(gen, (l * dk, dk), 1.0 / math.sqrt(l * dk))
    w_v = _draw(gen, (l * dv, dv), 1.0 / math.sqrt(l * dv))
    return pe_k, pe_v, w_k, w_v


def make_prefill(wl: PrefillWorkload, T: Optional[int] = None) -> Dict[str, torch.Tensor]:
    """Prefill inputs, all bf16 on the CPU.

    Draw order: q [B,T,H,dk], k [B,T,G,dk], v [B,T,G,dv], pe_k [l,dk],
    pe_v [l,dv], w_k [l*dk,dk], w_v [l*dv,dv], gates [B,T,H,3] (cmp, slc, win).
    ``T`` overrides the workload's length (ragged-tail parity cases).
    """
    T = wl.T if T is None else T
    gen = torch.Generator("cpu").manual_seed(wl.seed)
    q = _draw(gen, (wl.B, T, wl.H, wl.dk), 1.0)
    k = _draw(gen, (wl.B, T, wl.G, wl.dk), 1.0)
    v = _draw(gen, (wl.B, T, wl.G, wl.dv), 1.0)
    pe_k, pe_v, w_k, w_v = _phi_params(gen, wl.params.l, wl.dk, wl.dv)
    gates = _gates(gen, (wl.B, T, wl.H, 3))
    return dict(q=q, k=k, v=v, pe_k=pe_k, pe_v=pe_v, w_k=w_k, w_v=w_v, gates=gates)


def make_prefill_dout(wl: PrefillWorkload, T: Optional[int] = None) -> torch.Tensor:
    """Upstream gradient dout [B,T,H,dv] of the prefill output for the
    backward pass: bf16 N(0,1) from a generator of its own (seed + 1,000,003),
    so the forward inputs of ``make_prefill`` are unchanged."""
    T = wl.T if T is None else T
    gen = torch.Generator("cpu").manual_seed(wl.seed + 1_000_003)
    return _draw(gen, (wl.B, T, wl.H, wl.dv), 1.0)


def make_decode(wl: DecodeWorkload, B: Optional[int] = None, T: Optional[int] = None
                ) -> Dict[str, torch.Tensor]:
    """Decode inputs, all bf16 on the CPU.

    Draw order: kcache [B,G,T,dk], vcache [B,G,T,dv], q [B,H,dk], pe_k, pe_v,
    w_k, w_v, gates [B,H,3].  The caches are head-major so that one selection
    block of one KV head is one contiguous region.  The compressed caches are
    not drawn: they are computed from these caches by the compression step.
    """
    B = wl.B if B is None else B
    T = wl.T if T is None else T
    gen = torch.Generator("cpu").manual_seed(wl.seed)
    kcache = _draw(gen, (B, wl.G, T, wl.dk), 1.0)
    vcache = _draw(gen, (B, wl.G, T, wl.dv), 1.0)
    q = _draw(gen, (B, wl.H, wl.dk), 1.0)
    pe_k, pe_v, w_k, w_v = _phi_params(gen, wl.params.l, wl.dk, wl.dv)
    gates = _gates(gen, (B, wl.H, 3))
    return dict(kcache=kcache, vcache=vcache, q=q, pe_k=pe_k, pe_v=pe_v, w_k=w_k, w_v=w_v,
                gates=gates)


def make_decode_multi(wl: DecodeWorkload, m: int, B: Optional[int] = None, T: Optional[int] = None
                      ) -> Dict[str, torch.Tensor]:
    """Decode inputs with ``m`` query tokens per sequence (positions T-m ..
    T-1, all already in the caches), bf16 on the CPU.

    Draw order as ``make_decode`` with q [B,m,H,dk] and gates [B,m,H,3]; for
    m = 1 the values equal those of ``make_decode``.
    """
    B = wl.B if B is None else B
    T = wl.T if T is None else T
    gen = torch.Generator("cpu").manual_seed(wl.seed)
    kcache = _draw(gen, (B, wl.G, T, wl.dk), 1.0)
    vcache = _draw(gen, (B, wl.G, T, wl.dv), 1.0)
    q = _draw(gen, (B, m, wl.H, wl.dk), 1.0)
    pe_k, pe_v, w_k, w_v = _phi_params(gen, wl.params.l, wl.dk, wl.dv)
    gates = _gates(gen, (B, m, wl.H, 3))
    return dict(kcache=kcache, vcache=vcache, q=q, pe_k=pe_k, pe_v=pe_v, w_k=w_k, w_v=w_v,
                gates=gates)


def make_dsa(wl: DSAWorkload, B: Optional[int] = None, T: Optional[int] = None
             ) -> Dict[str, torch.Tensor]:
    """DSA decode inputs, all bf16 N(0,1) on the CPU.

    Draw order: qI [B,HI,dI], wI [B,HI], kI [B,T,dI], q [B,H,dk], k [B,T,dk],
    v [B,T,dv].
    """
    B = wl.B if B is None else B
    T = wl.T if T is None else T
    gen = torch.Generator("cpu").manual_seed(wl.seed)
    qI = _draw(gen, (B, wl.HI, wl.dI), 1.0)
    wI = _draw(gen, (B, wl.HI), 1.0)
    kI = _draw(gen, (B, T, wl.dI), 1.0)
    q = _draw(gen, (B, wl.H, wl.dk), 1.0)
    k = _draw(gen, (B, T, wl.dk), 1.0)
    v = _draw(gen, (B, T, wl.dv), 1.0)
    return dict(qI=qI, wI=wI, kI=kI, q=q, k=k, v=v)


def make_dsa_prefill(wl: DSAWorkload, B: Optional[int] = None, T: Optional[int] = None
                     ) -> Dict[str, torch.Tensor]:
    """DSA prefill inputs (every position is a query), all bf16 N(0,1) on the
    CPU.

    Draw order: qI [B,T,HI,dI], wI [B,T,HI], kI [B,T,dI], q [B,T,H,dk],
    k [B,T,dk], v [B,T,dv].
    """
    B = wl.B if B is None else B
    T = wl.T if T is None else T
    gen = torch.Generator("cpu").manual_seed(wl.seed)
    qI = _draw(gen, (B, T, wl.HI, wl.dI), 1.0)
    wI = _draw(gen, (B, T, wl.HI), 1.0)
    kI = _draw(gen, (B, T, wl.dI), 1.0)
    q = _draw(gen, (B, T, wl.H, wl.dk), 1.0)
    k = _draw(gen, (B, T, wl.dk), 1.0)
    v = _draw(gen, (B, T, wl.dv), 1.0)
    return dict(qI=qI, wI=wI, kI=kI, q=q, k=k, v=v)
