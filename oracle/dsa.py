"""fp64 oracle of the DSA-style indexed sparse decode step.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Page [P4] "딥시크 희소 어텐션 DSA 원리: 라이트닝 인덱서와 상위 2048 토큰 선택 구조 해설",
section "쉽게 이해하기" (easy explanation):
  * the lightning indexer scores every past token with a weighted sum over a
    few small heads of ReLU dot products, the keys being shared by all
    indexer heads:  I[s] = sum_h w_h * max(0, qI_h . kI_s);
  * the selector keeps the 2048 best positions and drops the rest
    (reading: ties go to the lower position; the decision is taken in fp32,
    the precision of the kernels);
  * attention then runs at full precision over the selected tokens only,
    with the softmax denominator summed over the selected set only
    (scale 1/sqrt(dk));
  * selection is made independently for each query position.
Key-message list of the same page: 2048 tokens are 1.6% of a 128k context.
"""
from __future__ import annotations

import math
from typing import Dict, Iterable, Optional

import numpy as np
import torch

from .nsa import to_f64

__all__ = ["dsa_indexer_scores", "topk_positions", "topk_alternatives", "topk_set_valid",
           "dsa_attention", "dsa_decode_reference", "dsa_prefill_reference"]


def dsa_indexer_scores(qI: np.ndarray, wI: np.ndarray, kI: np.ndarray) -> np.ndarray:
    """I[s] = sum_h w_h * ReLU(qI_h . kI_s) for every position s.

    qI [HI, dI], wI [HI], kI [T, dI] -> I [T] (fp64).
    """
    relu = np.maximum(kI @ qI.T, 0.0)          # [T, HI]
    return relu @ wI


def topk_positions(I32: np.ndarray, k: int) -> np.ndarray:
    """The k positions of largest fp32 score, ties to the lower position,
    returned ascending.  k >= T keeps every position."""
    T = I32.shape[0]
    if k >= T:
        return np.arange(T, dtype=np.int64)
    pos = np.arange(T)
    order = np.lexsort((pos, -I32.astype(np.float32)))
    return np.sort(order[:k])


def topk_alternatives(I32: np.ndarray, k: int, rel_tol: float):
    """(gap_rel, definite, band, need) for one row, as in the NSA selector:
    positions clearly above the cut must be kept, ``need`` more come from the
    band of positions within ``rel_tol`` of the cut."""
    T = I32.shape[0]
    if k >= T:
        return float("inf"), np.arange(T), np.zeros(0, dtype=np.int64), 0
    s = I32.astype(np.float64)
    order = np.lexsort((np.arange(T), -I32.astype(np.float32)))
    last_in, first_out = s[order[k - 1]], s[order[k]]
    cut = 0.5 * (last_in + first_out)
    scale = max(abs(last_in), abs(first_out), 1e-30)
    tol = rel_tol * scale
    above = np.nonzero(s > cut + tol)[0]
    band = np.nonzero(np.abs(s - cut) <= tol)[0]
    return (last_in - first_out) / scale, above, band, k - above.size


def topk_set_valid(I32: np.ndarray, kept, k: int, rel_tol: float):
    """Is ``kept`` (positions, any order) an acceptable top-k set of the row?

    Acceptable means: exactly min(k, T) distinct in-range positions, every
    position clearly above the cut kept, and the rest taken from the band of
    positions whose fp32 score lies within ``rel_tol`` (relative) of the cut
    (reading: near-ties may resolve either way).  Returns (ok, gap_rel).
    """
    T = I32.shape[0]
    kept = np.asarray(list(kept), dtype=np.int64)
    kset = set(kept.tolist())
    if len(kset) != kept.size or kept.size != min(k, T) or (kept.size and (kept.min() < 0 or kept.max() >= T)):
        return False, float("nan")
    gap, above, band, need = topk_alternatives(I32, k, rel_tol)
    a = set(above.tolist())
    extra = kset - a
    return bool(a <= kset and extra <= set(band.tolist()) and len(extra) == need), gap


def dsa_attention(q: np.ndarray, Ksel: np.ndarray, Vsel: np.ndarray, scale: float) -> np.ndarray:
    """Softmax attention of q [H, dk] over the selected keys only."""
    logits = (q @ Ksel.T) * scale
    logits = logits - logits.max(axis=-1, keepdims=True)
    e = np.exp(logits)
    return (e / e.sum(axis=-1, keepdims=True)) @ Vsel


def dsa_decode_reference(inp: Dict[str, torch.Tensor], topk: int,
                         batches: Optional[Iterable[int]] = None,
                         latent_dv: Optional[int] = None,
                         seq_lens: Optional[Iterable[int]] = None) -> Dict[str, np.ndarray]:
    """One DSA decode step for the batch rows ``batches`` (default all).

    inp: bf16 tensors of ``workloads.make_dsa``.  Row b's context holds
    T_b = seq_lens[b] tokens (default T): its query scores and keeps among
    positions s < T_b only.  Returns out [S,H,dv], idx [S,min(k,T)]
    (ascending, -1 past min(k,T_b)), I [S,T] fp64 and I32 [S,T] fp32 scores
    (zero past T_b).

    With ``inp["v"] is None`` the values are latent: value row s is the first
    ``latent_dv`` columns of key row s.  Same page, the paragraph that puts
    DSA on multi-head latent attention: one compressed latent vector is cached
    per token (its positional part kept as a separate stream), so keys and
    values are read from the same cached row.
    """
    qI, wI, kI, q, k = (inp[n] for n in ("qI", "wI", "kI", "q", "k"))
    v = inp.get("v")
    B, T, dk = k.shape
    H = q.shape[1]
    if v is None:
        if latent_dv is None or latent_dv > dk:
            raise ValueError("latent values need latent_dv <= dk")
        dv = latent_dv
    else:
        dv = v.shape[2]
    scale = 1.0 / math.sqrt(dk)
    batches = list(range(B)) if batches is None else list(batches)
    kk = min(topk, T)
    lens = [T] * B if seq_lens is None else [int(x) for x in seq_lens]
    res = dict(out=np.zeros((len(batches), H, dv)),
               idx=np.full((len(batches), kk), -1, dtype=np.int64),
               I=np.zeros((len(batches), T)), I32=np.zeros((len(batches), T), dtype=np.float32))
    for si, b in enumerate(batches):
        Tb = lens[b]
        assert 1 <= Tb <= T, "a row's context holds between 1 and T tokens"
        I = dsa_indexer_scores(to_f64(qI[b]), to_f64(wI[b]), to_f64(kI[b, :Tb]))
        I32 = I.astype(np.float32)
        sel = topk_positions(I32, topk)
        ti = torch.as_tensor(sel)
        Ksel = to_f64(k[b, ti])
        Vsel = Ksel[:, :dv] if v is None else to_f64(v[b, ti])
        res["out"][si] = dsa_attention(to_f64(q[b]), Ksel, Vsel, scale)
        res["idx"][si, :sel.size] = sel
        res["I"][si, :Tb], res["I32"][si, :Tb] = I, I32
    res["batches"] = np.array(batches)
    res["lens"] = np.array([lens[b] for b in batches])
    return res


def dsa_prefill_reference(inp: Dict[str, torch.Tensor], topk: int, b: int = 0,
                          rows: Optional[Iterable[int]] = None) -> Dict[str, np.ndarray]:
    """DSA over a whole sequence ``b``: every position t is a query.

    Same page, "쉽게 이해하기": the selection is made independently for each
    query position.  Readings taken for the prefill form:
      * the indexer query qI and weights wI belong to the query token, so
        inp holds them per position (``workloads.make_dsa_prefill``);
      * query t scores, keeps and attends over its causal prefix s <= t
        (t itself included), keeping min(topk, t + 1) positions.
    Returns out [R,H,dv] and, per row, the kept positions (a list of arrays,
    ascending) and the fp32 scores of the prefix.
    """
    qI, wI, kI, q, k, v = (inp[n] for n in ("qI", "wI", "kI", "q", "k", "v"))
    _, T, H, dk = q.shape
    dv = v.shape[2]
    scale = 1.0 / math.sqrt(dk)
    rows = list(range(T)) if rows is None else list(rows)
    kI_b, K, V = to_f64(kI[b]), to_f64(k[b]), to_f64(v[b])
    out = np.zeros((len(rows), H, dv))
    idx, I32s = [], []
    for r, t in enumerate(rows):
        I = dsa_indexer_scores(to_f64(qI[b, t]), to_f64(wI[b, t]), kI_b[: t + 1])
        I32 = I.astype(np.float32)
        sel = topk_positions(I32, topk)
        out[r] = dsa_attention(to_f64(q[b, t]), K[sel], V[sel], scale)
        idx.append(sel)
        I32s.append(I32)
    return dict(out=out, idx=idx, I32=I32s, rows=np.array(rows))
