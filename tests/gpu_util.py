"""Helpers shared by the GPU parity tests (device transfer, comparison rules)."""
import numpy as np
import torch

from oracle import nsa as O


def to_dev(inp, keys=None):
    keys = keys or list(inp)
    return {k: inp[k].to("cuda") for k in keys}


def bf16_compare(got: torch.Tensor, exact: np.ndarray, absmag: np.ndarray, acc_rel: float = 2.0 ** -20):
    """Compare a bf16 kernel output with the oracle's exact (pre-rounding) fp64
    values of a dot product.  The oracle rounds the exact value; the kernel
    rounds its fp32 accumulation, whose error is bounded by
    ``acc_rel * absmag`` (absmag = sum of |terms| of the dot product; fp32
    accumulation of a few thousand terms stays well inside 2**-20 of it).
    Allowed: |got - exact| <= half a bf16 step of ``exact`` + that bound.
    Returns the number of elements that differ from the oracle's rounding."""
    g = got.detach().cpu().to(torch.float64).numpy().reshape(exact.shape)
    want = O.bf16_round(exact)
    nd = int((g != want).sum())
    _, ee = np.frexp(np.maximum(np.abs(exact), 1e-300))
    half = np.ldexp(1.0, ee - 9)
    allow = half * (1 + 1e-9) + acc_rel * absmag
    bad = np.abs(g - exact) > allow
    worst = np.argsort((np.abs(g - exact) / allow).ravel())[-3:]
    print(f"bf16_compare: {nd} of {exact.size} differ from the oracle's rounding; worst "
          f"(got, exact, allow): {[(g.ravel()[i], exact.ravel()[i], allow.ravel()[i]) for i in worst]}")
    assert not bad.any(), f"{int(bad.sum())} elements outside the bound"
    assert np.isfinite(g).all()
    return nd


def compress_exact(inp, B, G, layout_btgd, kname, pename, wname, seqs=None):
    """Oracle's exact (pre-rounding) compressed values [S,G,Nc,d] of the
    sequences ``seqs`` (default all B) and, for the tolerance of
    ``bf16_compare``, the sum of the absolute values of each dot product's
    terms."""
    pe, w = O.to_f64(inp[pename]), O.to_f64(inp[wname])
    seqs = list(range(B)) if seqs is None else list(seqs)
    out, mag = [], []
    for b in seqs:
        for g in range(G):
            X = O.to_f64(inp[kname][b, :, g] if layout_btgd else inp[kname][b, g])
            out.append(O.compress(X, pe, w, 32, 16, round_bf16=False))
            Nc = out[-1].shape[0]
            flat = np.abs(np.stack([(X[16 * i: 16 * i + 32] + pe).reshape(-1) for i in range(Nc)])) \
                if Nc else np.zeros((0, w.shape[0]))
            mag.append(flat @ np.abs(w))
    sh = out[0].shape
    return np.stack(out).reshape(len(seqs), G, *sh), np.stack(mag).reshape(len(seqs), G, *sh)


def cache_f64(t: torch.Tensor) -> np.ndarray:
    """A bf16 device cache as fp64 numpy (exact): what the oracle is handed
    when it scores the GPU's own compressed cache."""
    return t.detach().float().cpu().numpy().astype(np.float64)
