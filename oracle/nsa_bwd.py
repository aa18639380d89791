"""fp64 oracle of the NSA backward pass: the gradients of the forward defined
in ``oracle.nsa`` with respect to every input.

TEST INFRASTRUCTURE ONLY (see the package docstring): never imported by the
product package.

The pages quote a 6.0x faster backward pass than full attention at 64k
[P2 section III.3, training speed-up] but give no formula for it, so the
gradients here are those of the forward of ``oracle.nsa`` (compression,
compressed / selected / window attention, gated combine), under these
readings:

  B1  The kept blocks are constants.  Top-n is a discrete choice and has no
      gradient, so the backward uses the forward's selection ``idx`` and the
      block scores receive no gradient.
  B2  The bf16 rounding of the compressed cache passes gradients unchanged
      (straight-through): dKc, dVc flow to the exact fp64 value of the
      compression map.
  B3  The gates are inputs, as in the forward; their gradient is returned.
      The compression map W_c and position embedding PE are shared by the KV
      heads, so their gradients sum over the groups.

Given dout = dLoss/dout [T, H, dv], the oracle returns dq, dk, dv, dgates and
the gradients of W_cK, W_cV, PE_K, PE_V, all in fp64.

Every branch is softmax attention.  Per query row, with s = scale * q K^T,
P = softmax(s) over the branch's keys and O = P V, its backward is the
textbook one:
    dV_j += P_j dO                   dP_j = dO . V_j
    dS_j  = P_j (dP_j - dO . O)      dq  += scale * sum_j dS_j K_j
    dK_j += scale * dS_j q
The gated combine out = g_c O_cmp + g_s O_slc + g_w O_win gives each branch
dO = g * dout and dg = dout . O_branch.  The compression map
Xc_i = flatten(X[d*i : d*i+l] + PE) @ W gives
    dW += flatten(X[d*i : d*i+l] + PE)^T dXc_i,   dB_i = dXc_i W^T as [l, dX],
    dPE += dB_i,   dX[d*i + r] += dB_i[r].

Parity: pinned in ``tests/test_oracle_backward.py`` by central finite
differences of <dout, out> along random directions (through
``nsa_prefill_forward_fixed``, the forward with the selection held fixed and
the cache unrounded), by an independent torch-autograd formulation, and by
special cases (one visible key gives dq = 0; dout = 0 gives zero gradients).
"""
from __future__ import annotations

import math
from typing import Dict, Optional

import numpy as np
import torch

from workloads import NSAParams

from .nsa import compress, nsa_group_rows, num_visible_compressed, selected_keys, to_f64

__all__ = ["attend_bwd", "compress_bwd", "nsa_group_bwd", "nsa_prefill_backward",
           "nsa_prefill_forward_fixed"]


def attend_bwd(q: np.ndarray, K: np.ndarray, V: np.ndarray, keys: np.ndarray, scale: float,
               dO: np.ndarray):
    """Softmax attention of q [hh, dk] over K[keys], V[keys] and its backward
    for the upstream gradient dO [hh, dv].

    Returns (O [hh, dv], dq [hh, dk], dK [n, dk], dV [n, dv]) where dK, dV
    are the gradients of the rows K[keys], V[keys].  An empty key set gives
    O = 0 and no gradient (the empty-branch reading of the forward).
    """
    hh, dk = q.shape
    dv = V.shape[1]
    if keys.size == 0:
        return np.zeros((hh, dv)), np.zeros((hh, dk)), np.zeros((0, dk)), np.zeros((0, dv))
    Kk, Vk = K[keys], V[keys]
    s = (q @ Kk.T) * scale
    s = s - s.max(axis=-1, keepdims=True)
    e = np.exp(s)
    P = e / e.sum(axis=-1, keepdims=True)            # [hh, n]
    O = P @ Vk                                        # [hh, dv]
    dP = dO @ Vk.T                                    # [hh, n]
    dS = P * (dP - (dO * O).sum(axis=-1, keepdims=True))
    dq = scale * (dS @ Kk)
    dKk = scale * (dS.T @ q)
    dVk = P.T @ dO
    return O, dq, dKk, dVk


def compress_bwd(X: np.ndarray, PE: np.ndarray, W: np.ndarray, l: int, d: int,
                 dXc: np.ndarray):
    """Backward of the compression map [P2 II.1, P3 token compression]
    Xc_i = flatten(X[d*i : d*i+l] + PE) @ W for the gradient dXc [Nc, dout].

    Returns (dX [T, dX], dPE [l, dX], dW [l*dX, dout]).
    """
    T, dx = X.shape
    Nc = dXc.shape[0]
    dX = np.zeros_like(X)
    dPE = np.zeros_like(PE)
    dW = np.zeros_like(W)
    if Nc == 0:
        return dX, dPE, dW
    flat = np.stack([(X[d * i: d * i + l] + PE).reshape(l * dx) for i in range(Nc)])
    dW = flat.T @ dXc
    dB = (dXc @ W.T).reshape(Nc, l, dx)
    dPE = dB.sum(axis=0)
    starts = d * np.arange(Nc)
    for r in range(l):
        np.add.at(dX, starts + r, dB[:, r])
    return dX, dPE, dW


def nsa_group_bwd(q: np.ndarray, t_rows: np.ndarray, K: np.ndarray, V: np.ndarray,
                  Kc: np.ndarray, Vc: np.ndarray, gates: np.ndarray, idx: np.ndarray,
                  params: NSAParams, scale: float, dout: np.ndarray) -> Dict[str, np.ndarray]:
    """Backward of the three branches and the gated combine for the rows
    ``t_rows`` of one sequence and one KV group, the kept blocks fixed to
    ``idx`` (reading B1).

    q [R, hh, dk], K [T, dk], V [T, dv], Kc [Nc, dk], Vc [Nc, dv] (the values
    the forward attended to), gates [R, hh, 3], idx [R, n], dout [R, hh, dv].
    Returns dq [R, hh, dk], dK [T, dk], dV [T, dv] (selected and window
    branches), dKc [Nc, dk], dVc [Nc, dv] (compressed branch), dgates
    [R, hh, 3] and out [R, hh, dv].
    """
    p_ = params
    R, hh, dk = q.shape
    dv = V.shape[1]
    Nc = Kc.shape[0]
    dq = np.zeros_like(q)
    dK = np.zeros_like(K)
    dV = np.zeros_like(V)
    dKc = np.zeros_like(Kc)
    dVc = np.zeros_like(Vc)
    dg = np.zeros((R, hh, 3))
    out = np.zeros((R, hh, dv))
    for r in range(R):
        t = int(t_rows[r])
        branches = (
            (Kc, Vc, np.arange(int(num_visible_compressed(t, p_.l, p_.d, Nc))) if Nc else np.zeros(0, np.int64),
             dKc, dVc),
            (K, V, selected_keys(idx[r], t, p_.lsel), dK, dV),
            (K, V, np.arange(max(0, t - p_.w + 1), t + 1), dK, dV),
        )
        for bi, (Kb, Vb, keys, dKb, dVb) in enumerate(branches):
            g = gates[r, :, bi:bi + 1]
            O, dqb, dKk, dVk = attend_bwd(q[r], Kb, Vb, keys, scale, g * dout[r])
            out[r] += g * O
            dg[r, :, bi] = (dout[r] * O).sum(axis=-1)
            dq[r] += dqb
            if keys.size:
                np.add.at(dKb, keys, dKk)
                np.add.at(dVb, keys, dVk)
    return dict(dq=dq, dK=dK, dV=dV, dKc=dKc, dVc=dVc, dgates=dg, out=out)


def _inputs_f64(inp: Dict[str, torch.Tensor], b: int):
    return dict(q=to_f64(inp["q"][b]), k=to_f64(inp["k"][b]), v=to_f64(inp["v"][b]),
                gates=to_f64(inp["gates"][b]), pe_k=to_f64(inp["pe_k"]), pe_v=to_f64(inp["pe_v"]),
                w_k=to_f64(inp["w_k"]), w_v=to_f64(inp["w_v"]))


def nsa_prefill_backward(inp: Dict[str, torch.Tensor], dout: np.ndarray, b: int = 0,
                         params: NSAParams = NSAParams(),
                         idx: Optional[np.ndarray] = None,
                         round_cache: bool = True) -> Dict[str, np.ndarray]:
    """Gradients of <dout, out> for every row of sequence ``b``.

    inp: the bf16 tensors of ``workloads.make_prefill``; dout [T, H, dv]
    fp64.  idx [T, G, n]: the forward's kept blocks (computed here by the
    forward oracle when None).  The attention backward runs on the cache the
    forward reads (bf16-rounded); ``round_cache=False`` uses its exact value
    instead, the differentiable function of ``nsa_prefill_forward_fixed``.
    Returns dq [T, H, dk], dk [T, G, dk],
    dv [T, G, dv], dgates [T, H, 3], dw_k, dw_v, dpe_k, dpe_v, the forward
    out [T, H, dv] and idx, and the compressed cache's gradients dkc
    [G, Nc, dk], dvc [G, Nc, dv] (what the compression map's backward
    receives).
    """
    x = _inputs_f64(inp, b)
    T, H, dk = x["q"].shape
    G = x["k"].shape[1]
    dv = x["v"].shape[2]
    hpg = H // G
    scale = 1.0 / math.sqrt(dk)
    rows = np.arange(T)
    res = dict(dq=np.zeros((T, H, dk)), dk=np.zeros((T, G, dk)), dv=np.zeros((T, G, dv)),
               dgates=np.zeros((T, H, 3)), dw_k=np.zeros_like(x["w_k"]), dw_v=np.zeros_like(x["w_v"]),
               dpe_k=np.zeros_like(x["pe_k"]), dpe_v=np.zeros_like(x["pe_v"]),
               out=np.zeros((T, H, dv)), idx=np.zeros((T, G, params.n), dtype=np.int32))
    for g in range(G):
        K, V = x["k"][:, g], x["v"][:, g]
        Kc = compress(K, x["pe_k"], x["w_k"], params.l, params.d, round_bf16=round_cache)
        Vc = compress(V, x["pe_v"], x["w_v"], params.l, params.d, round_bf16=round_cache)
        hs = slice(g * hpg, (g + 1) * hpg)
        if idx is None:
            ig = nsa_group_rows(x["q"][:, hs], rows, K, V, Kc, Vc, x["gates"][:, hs], params, scale)["idx"]
        else:
            ig = idx[:, g]
        r = nsa_group_bwd(x["q"][:, hs], rows, K, V, Kc, Vc, x["gates"][:, hs], ig, params, scale,
                          dout[:, hs])
        dKx, dpk, dwk = compress_bwd(K, x["pe_k"], x["w_k"], params.l, params.d, r["dKc"])
        dVx, dpv, dwv = compress_bwd(V, x["pe_v"], x["w_v"], params.l, params.d, r["dVc"])
        res.setdefault("dkc", []).append(r["dKc"])
        res.setdefault("dvc", []).append(r["dVc"])
        res["dq"][:, hs] = r["dq"]
        res["dk"][:, g] = r["dK"] + dKx
        res["dv"][:, g] = r["dV"] + dVx
        res["dgates"][:, hs] = r["dgates"]
        res["dw_k"] += dwk
        res["dw_v"] += dwv
        res["dpe_k"] += dpk
        res["dpe_v"] += dpv
        res["out"][:, hs] = r["out"]
        res["idx"][:, g] = ig
    res["dkc"] = np.stack(res["dkc"])
    res["dvc"] = np.stack(res["dvc"])
    return res


def nsa_prefill_forward_fixed(x: Dict[str, np.ndarray], idx: np.ndarray, params: NSAParams,
                              round_cache: bool = False) -> np.ndarray:
    """The forward of ``oracle.nsa`` for one sequence with the kept blocks
    fixed to ``idx`` [T, G, n], on fp64 inputs ``x`` (keys as in
    ``_inputs_f64``).  ``round_cache=False`` keeps the compressed cache at its
    exact fp64 value, the function whose gradient readings B1/B2 describe.
    Returns out [T, H, dv].
    """
    from .nsa import cmp_attention, sel_attention, win_attention
    q = x["q"]
    T, H, dk = q.shape
    G = x["k"].shape[1]
    dv = x["v"].shape[2]
    hpg = H // G
    scale = 1.0 / math.sqrt(dk)
    out = np.zeros((T, H, dv))
    rows = np.arange(T)
    for g in range(G):
        K, V = x["k"][:, g], x["v"][:, g]
        Kc = compress(K, x["pe_k"], x["w_k"], params.l, params.d, round_bf16=round_cache)
        Vc = compress(V, x["pe_v"], x["w_v"], params.l, params.d, round_bf16=round_cache)
        hs = slice(g * hpg, (g + 1) * hpg)
        gt = x["gates"][:, hs]
        oc, _ = cmp_attention(q[:, hs], rows, Kc, Vc, scale, params.l, params.d)
        for t in range(T):
            os_ = sel_attention(q[t, hs], t, K, V, idx[t, g], params.lsel, scale)
            ow = win_attention(q[t, hs], t, K, V, params.w, scale)
            out[t, hs] = gt[t, :, 0:1] * oc[t] + gt[t, :, 1:2] * os_ + gt[t, :, 2:3] * ow
    return out
