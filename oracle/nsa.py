"""fp64 oracle of the Native Sparse Attention (NSA) forward pass.

TEST INFRASTRUCTURE ONLY (see the package docstring): never imported by the
product package.

What it computes, step by step, for one sequence and one KV group g whose
query heads are h = g*hpg .. g*hpg+hpg-1 (hpg = H/G query heads per KV head):

 1. Token compression [P2 section II, P3 token-compression paragraph]:
    blocks of l consecutive keys at stride d, each block plus an intra-block
    position embedding flattened and mapped by one linear map W_c to one
    vector.  Nc = floor((T-l)/d) + 1 blocks.  The compressed keys/values are
    a cache and are stored in bf16: the oracle rounds the exact value once.
 2. Compressed attention [P2 II.1, P3]: query t attends to every compressed
    block whose last token is <= t (a block is visible only when complete),
    softmax with scale 1/sqrt(dk).  Nothing visible -> output 0.
 3. Block importance [P3 token-selection paragraph: importance of each block
    is derived from the compressed tokens; selection is per GQA group, P1
    hardware-aware design + P2 IV.2]:  S[t,j] = sum over heads of the group
    of sum_i w(i,j) p[t,h,i], where w(i,j) is the number of d-token chunks
    that compressed block i and selection block j share.
 4. Top-n selection [P2 II: n=16 blocks of l'=64, 1 initial + 2 local
    blocks included]: blocks 0, j_t and j_t-1 (j_t = floor(t/l')) are always
    kept; the other n-3 are the highest-scoring causal blocks, ties to the
    lower index.  If the query has at most n causal blocks, all are kept.
 5. Selected attention over the original tokens s <= t of the kept blocks
    [P2 II.2, P3]; sliding-window attention over the last w tokens
    (t-w, t] [P2 II.3, P3 sliding-window paragraph].  Each branch has its
    own softmax with scale 1/sqrt(dk).
 6. The three paths are combined with per-head gates
    out = g_cmp*O_cmp + g_slc*O_slc + g_win*O_win  (the pages only say the
    three paths run in parallel [P2 II]; gates are given inputs).

Decode is row t = T-1 of the same definition, read from the caches.
"""
from __future__ import annotations

import math
from typing import Dict, Iterable, List, Optional, Sequence

import numpy as np
import torch

from workloads import NSAParams

__all__ = [
    "to_f64", "bf16_round", "num_compressed", "num_visible_compressed",
    "compress", "cmp_attention", "overlap_matrix", "block_scores",
    "select_blocks", "selection_alternatives", "selection_set_valid", "selected_keys", "sel_attention",
    "win_attention", "nsa_group_rows", "nsa_prefill_reference",
    "nsa_decode_reference", "nsa_decode_multi_reference", "decode_tokens_read",
]


def to_f64(t: torch.Tensor) -> np.ndarray:
    """bf16 (or any float) torch tensor -> numpy fp64 (exact for bf16)."""
    return t.detach().cpu().to(torch.float64).numpy()


def bf16_round(x) -> np.ndarray:
    """Round fp64 values to the nearest bf16 value, ties to even.

    bf16 keeps 8 significant bits; below 2**-126 its grid is the subnormal
    grid of spacing 2**-133.  Returned as fp64 values lying on the bf16 grid.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros_like(x)
    nz = x != 0
    _, e = np.frexp(x[nz])                 # |x| = m * 2**e, 0.5 <= m < 1
    e = np.maximum(e, -125)                # subnormal range keeps the 2**-133 spacing
    q = np.rint(np.ldexp(x[nz], 8 - e))    # integer in [128, 256]: ties to even
    out[nz] = np.ldexp(q, e - 8)
    return out


def num_compressed(T: int, l: int = 32, d: int = 16) -> int:
    """Number of compression blocks: windows [d*i, d*i+l) inside [0, T)."""
    return 0 if T < l else (T - l) // d + 1


def num_visible_compressed(t, l: int, d: int, Nc: int):
    """|C_t|: blocks i whose last token d*i+l-1 is <= t (reading: a block is
    visible only when complete)."""
    t = np.asarray(t, dtype=np.int64)
    n = np.where(t >= l - 1, (t - (l - 1)) // d + 1, 0)
    return np.minimum(n, Nc)


def compress(X: np.ndarray, PE: np.ndarray, W: np.ndarray, l: int, d: int,
             round_bf16: bool = True) -> np.ndarray:
    """Token compression [P2 II.1, P3].

    X [T, dX] keys (or values) of one KV head, PE [l, dX] intra-block position
    embedding, W [l*dX, dout].  Block i = flatten(X[d*i : d*i+l] + PE) @ W,
    rounded once to bf16 (the compressed cache is stored in bf16);
    ``round_bf16=False`` returns the exact fp64 value before that rounding.
    """
    T, dX = X.shape
    Nc = num_compressed(T, l, d)
    if Nc == 0:
        return np.zeros((0, W.shape[1]))
    flat = np.stack([(X[d * i: d * i + l] + PE).reshape(l * dX) for i in range(Nc)])
    exact = flat @ W
    return bf16_round(exact) if round_bf16 else exact


def _softmax_masked(logits: np.ndarray, valid: np.ndarray) -> np.ndarray:
    """softmax over the entries where ``valid``; all-invalid rows give 0."""
    z = np.where(valid, logits, -np.inf)
    m = z.max(axis=-1, keepdims=True)
    m = np.where(np.isfinite(m), m, 0.0)
    e = np.where(valid, np.exp(np.where(valid, z - m, 0.0)), 0.0)
    den = e.sum(axis=-1, keepdims=True)
    return np.where(den > 0, e / np.where(den > 0, den, 1.0), 0.0)


def cmp_attention(q: np.ndarray, t: np.ndarray, Kc: np.ndarray, Vc: np.ndarray,
                  scale: float, l: int, d: int):
    """Compressed attention [P2 II.1, P3 token compression].

    q [R, hh, dk] queries of rows t [R]; Kc [Nc, dk], Vc [Nc, dv].
    Returns (O [R, hh, dv], p [R, hh, Nc]) with p = 0 on invisible blocks.
    """
    Nc = Kc.shape[0]
    if Nc == 0:                      # no complete block anywhere: empty branch -> 0
        return np.zeros(q.shape[:2] + (Vc.shape[1],)), np.zeros(q.shape[:2] + (0,))
    n_t = num_visible_compressed(t, l, d, Nc)
    logits = (q @ Kc.T) * scale                             # [R, hh, Nc]
    valid = (np.arange(Nc)[None, :] < n_t[:, None])[:, None, :]
    p = _softmax_masked(logits, np.broadcast_to(valid, logits.shape))
    return p @ Vc, p


def overlap_matrix(Nc: int, nb: int, l: int, d: int, lsel: int) -> np.ndarray:
    """w(i, j) = |[d*i, d*i+l) intersect [lsel*j, lsel*j+lsel)| / d: the number of
    d-token chunks shared by compressed block i and selection block j
    (reading of 'importance from the compressed tokens', P3)."""
    i = np.arange(Nc)[:, None]
    j = np.arange(nb)[None, :]
    lo = np.maximum(d * i, lsel * j)
    hi = np.minimum(d * i + l, lsel * j + lsel)
    return np.maximum(hi - lo, 0).astype(np.float64) / d


def block_scores(p: np.ndarray, nb: int, l: int, d: int, lsel: int) -> np.ndarray:
    """S[r, j] = sum_h sum_i w(i,j) p[r,h,i]  (head sum over one GQA group).

    p [R, hh, Nc] -> S [R, nb] in fp64.
    """
    Om = overlap_matrix(p.shape[-1], nb, l, d, lsel)
    return np.einsum("rhi,ij->rj", p, Om)


def select_blocks(S32: np.ndarray, t: int, n: int, lsel: int) -> np.ndarray:
    """Top-n block selection for one query row [P2 II: n=16 incl. 1 initial and
    2 local blocks].

    S32: the row's block scores as fp32 (the decision is taken in the fp32
    precision of the kernels).  Blocks 0, j_t, j_t-1 are forced; the remaining
    n-|F| come from the other causal blocks ordered by (-S, j): higher score
    first, ties to the lower index.  Returned ascending, padded with -1.
    """
    jt = t // lsel
    out = np.full(n, -1, dtype=np.int32)
    if jt + 1 <= n:
        out[: jt + 1] = np.arange(jt + 1)
        return out
    forced = np.array(sorted({0, jt, jt - 1}), dtype=np.int64)
    cand = np.setdiff1d(np.arange(jt + 1), forced)
    order = np.lexsort((cand, -S32[cand].astype(np.float32)))
    chosen = cand[order[: n - forced.size]]
    out[:] = np.sort(np.concatenate([forced, chosen]))
    return out


def selection_alternatives(S32: np.ndarray, t: int, n: int, lsel: int, rel_tol: float):
    """Near-tie bookkeeping for one row.

    Returns (gap_rel, definite, band, need): gap_rel is the relative fp32
    score gap between the last kept and the first dropped free block (inf if
    no real choice is made); every block of ``definite`` (forced blocks and
    free blocks scoring clearly above the cut) must be selected; ``need``
    more blocks must come from ``band``, the free blocks whose score lies
    within ``rel_tol`` (relative) of the cut value.
    """
    jt = t // lsel
    if jt + 1 <= n:
        return float("inf"), set(range(jt + 1)), set(), 0
    forced = {0, jt, jt - 1}
    cand = np.array(sorted(set(range(jt + 1)) - forced), dtype=np.int64)
    s = S32[cand].astype(np.float64)
    order = np.lexsort((cand, -S32[cand].astype(np.float32)))
    kfree = n - len(forced)
    last_in = s[order[kfree - 1]]
    first_out = s[order[kfree]] if cand.size > kfree else -np.inf
    if not np.isfinite(first_out):
        return float("inf"), forced | set(cand.tolist()), set(), 0
    cut = 0.5 * (last_in + first_out)
    scale = max(abs(last_in), abs(first_out), 1e-30)
    gap = (last_in - first_out) / scale
    tol = rel_tol * scale
    above = set(cand[s > cut + tol].tolist())
    band = set(cand[np.abs(s - cut) <= tol].tolist())
    return gap, forced | above, band, kfree - len(above)


def selection_set_valid(S32: np.ndarray, t: int, row, n: int, lsel: int, rel_tol: float):
    """Is the index row ``row`` (n entries, ascending, -1 padded) an acceptable
    selection for query t?  Acceptable means: the kept blocks ascending and
    distinct in front, -1 after them, the forced and clearly-above-the-cut
    blocks all kept, and the remaining picks taken from the near-tie band of
    ``selection_alternatives``.  Returns (ok, gap_rel)."""
    row = [int(j) for j in row]
    kept = [j for j in row if j >= 0]
    if row[: len(kept)] != sorted(set(kept)) or any(j != -1 for j in row[len(kept):]):
        return False, float("nan")
    gap, definite, band, need = selection_alternatives(S32, t, n, lsel, rel_tol)
    ks = set(kept)
    extra = ks - definite
    return bool(definite <= ks and extra <= band and len(extra) == need), gap


def selected_keys(blocks: Sequence[int], t: int, lsel: int) -> np.ndarray:
    """Token positions s <= t inside the kept blocks (ascending)."""
    parts = [np.arange(j * lsel, min(j * lsel + lsel, t + 1)) for j in blocks if j >= 0]
    parts = [p for p in parts if p.size]
    return np.concatenate(parts) if parts else np.zeros(0, dtype=np.int64)


def _attend(q: np.ndarray, K: np.ndarray, V: np.ndarray, keys: np.ndarray, scale: float):
    """Textbook softmax attention of q [hh, dk] over K[keys], V[keys]."""
    if keys.size == 0:
        return np.zeros((q.shape[0], V.shape[1]))
    logits = (q @ K[keys].T) * scale
    logits = logits - logits.max(axis=-1, keepdims=True)
    e = np.exp(logits)
    return (e / e.sum(axis=-1, keepdims=True)) @ V[keys]


def sel_attention(q, t, K, V, blocks, lsel, scale):
    """Selected-block attention [P2 II.2, P3 token selection]: original tokens
    s <= t of the kept blocks, own softmax."""
    return _attend(q, K, V, selected_keys(blocks, t, lsel), scale)


def win_attention(q, t, K, V, w, scale):
    """Sliding-window attention [P2 II.3, P3]: tokens s in (t-w, t]."""
    return _attend(q, K, V, np.arange(max(0, t - w + 1), t + 1), scale)


def nsa_group_rows(q: np.ndarray, t_rows: np.ndarray, K: np.ndarray, V: np.ndarray,
                   Kc: np.ndarray, Vc: np.ndarray, gates: np.ndarray, params: NSAParams,
                   scale: float, chunk: int = 128) -> Dict[str, np.ndarray]:
    """All three branches for the rows ``t_rows`` of one sequence and one KV group.

    q [R, hh, dk], K [T, dk], V [T, dv] (this group's keys/values),
    Kc [Nc, dk], Vc [Nc, dv], gates [R, hh, 3] (cmp, slc, win).
    """
    p_ = params
    T = K.shape[0]
    nb = -(-T // p_.lsel)
    R, hh, _ = q.shape
    dv = V.shape[1]
    o_cmp = np.zeros((R, hh, dv))
    o_slc = np.zeros((R, hh, dv))
    o_win = np.zeros((R, hh, dv))
    S = np.zeros((R, nb))
    idx = np.zeros((R, p_.n), dtype=np.int32)
    for r0 in range(0, R, chunk):
        r1 = min(R, r0 + chunk)
        oc, pc = cmp_attention(q[r0:r1], t_rows[r0:r1], Kc, Vc, scale, p_.l, p_.d)
        o_cmp[r0:r1] = oc
        S[r0:r1] = block_scores(pc, nb, p_.l, p_.d, p_.lsel)
    S32 = S.astype(np.float32)
    for r in range(R):
        t = int(t_rows[r])
        idx[r] = select_blocks(S32[r], t, p_.n, p_.lsel)
        o_slc[r] = sel_attention(q[r], t, K, V, idx[r], p_.lsel, scale)
        o_win[r] = win_attention(q[r], t, K, V, p_.w, scale)
    out = gates[..., 0:1] * o_cmp + gates[..., 1:2] * o_slc + gates[..., 2:3] * o_win
    return dict(out=out, o_cmp=o_cmp, o_slc=o_slc, o_win=o_win, S=S, S32=S32, idx=idx)


def nsa_prefill_reference(inp: Dict[str, torch.Tensor], rows: Optional[Iterable[int]] = None,
                          b: int = 0, params: NSAParams = NSAParams(),
                          kc: Optional[np.ndarray] = None, vc: Optional[np.ndarray] = None
                          ) -> Dict[str, np.ndarray]:
    """Prefill forward for sequence ``b`` at query rows ``rows`` (default all).

    inp: the bf16 tensors of ``workloads.make_prefill``.  kc/vc: optional
    compressed caches [G, Nc, d] (fp64 on the bf16 grid); computed here when
    absent.  Returns out/o_cmp/o_slc/o_win [R, H, dv], idx [R, G, n],
    S and S32 [R, G, nb], kc [G, Nc, dk], vc [G, Nc, dv].
    """
    q_t, k_t, v_t = inp["q"], inp["k"], inp["v"]
    _, T, H, dk = q_t.shape
    G = k_t.shape[2]
    dv = v_t.shape[3]
    hpg = H // G
    scale = 1.0 / math.sqrt(dk)
    rows = np.arange(T) if rows is None else np.asarray(list(rows), dtype=np.int64)
    pe_k, pe_v = to_f64(inp["pe_k"]), to_f64(inp["pe_v"])
    w_k, w_v = to_f64(inp["w_k"]), to_f64(inp["w_v"])
    gates = to_f64(inp["gates"][b, torch.as_tensor(rows)])               # [R, H, 3]
    qr = to_f64(q_t[b, torch.as_tensor(rows)])                           # [R, H, dk]
    nb = -(-T // params.lsel)
    R = rows.size
    res = dict(out=np.zeros((R, H, dv)), o_cmp=np.zeros((R, H, dv)),
               o_slc=np.zeros((R, H, dv)), o_win=np.zeros((R, H, dv)),
               idx=np.zeros((R, G, params.n), dtype=np.int32),
               S=np.zeros((R, G, nb)), S32=np.zeros((R, G, nb), dtype=np.float32))
    kcs, vcs = [], []
    for g in range(G):
        K = to_f64(k_t[b, :, g, :])
        V = to_f64(v_t[b, :, g, :])
        Kc = compress(K, pe_k, w_k, params.l, params.d) if kc is None else kc[g]
        Vc = compress(V, pe_v, w_v, params.l, params.d) if vc is None else vc[g]
        kcs.append(Kc)
        vcs.append(Vc)
        hs = slice(g * hpg, (g + 1) * hpg)
        r = nsa_group_rows(qr[:, hs], rows, K, V, Kc, Vc, gates[:, hs], params, scale)
        for key in ("out", "o_cmp", "o_slc", "o_win"):
            res[key][:, hs] = r[key]
        res["idx"][:, g] = r["idx"]
        res["S"][:, g] = r["S"]
        res["S32"][:, g] = r["S32"]
    res["kc"] = np.stack(kcs)
    res["vc"] = np.stack(vcs)
    res["rows"] = rows
    return res


def nsa_decode_reference(inp: Dict[str, torch.Tensor], seqs: Optional[Iterable[int]] = None,
                         params: NSAParams = NSAParams(),
                         kc: Optional[np.ndarray] = None, vc: Optional[np.ndarray] = None,
                         seq_lens: Optional[Sequence[int]] = None) -> Dict[str, np.ndarray]:
    """Single-token decode for the sequences ``seqs`` (default all).

    inp: the bf16 tensors of ``workloads.make_decode`` (caches [B,G,T,d],
    q [B,H,dk], gates [B,H,3]).  Sequence b holds len_b = seq_lens[b] tokens
    (default T, the cache capacity); its query is at position t = len_b - 1
    (the cache already holds the new token) and only cache rows < len_b exist
    for it.  kc/vc: optional compressed caches [B,G,Nc,d] (fp64) at capacity;
    a sequence uses the entries that lie inside its own tokens (entry i only
    depends on tokens 16i .. 16i+31).  Computed here when absent.  Returns
    out [S,H,dv], idx [S,G,n], S32 [S,G,nb], kc/vc [S,G,Nc,d] (nb, Nc at
    capacity; a shorter sequence's rows are zero past its own).
    """
    kcache, vcache, q_t = inp["kcache"], inp["vcache"], inp["q"]
    B, G, T, dk = kcache.shape
    H = q_t.shape[1]
    dv = vcache.shape[3]
    hpg = H // G
    scale = 1.0 / math.sqrt(dk)
    seqs = list(range(B)) if seqs is None else list(seqs)
    lens = [T] * B if seq_lens is None else [int(x) for x in seq_lens]
    pe_k, pe_v = to_f64(inp["pe_k"]), to_f64(inp["pe_v"])
    w_k, w_v = to_f64(inp["w_k"]), to_f64(inp["w_v"])
    nb = -(-T // params.lsel)
    Nc = num_compressed(T, params.l, params.d)
    S_ = len(seqs)
    res = dict(out=np.zeros((S_, H, dv)), o_cmp=np.zeros((S_, H, dv)),
               o_slc=np.zeros((S_, H, dv)), o_win=np.zeros((S_, H, dv)),
               idx=np.zeros((S_, G, params.n), dtype=np.int32),
               S=np.zeros((S_, G, nb)), S32=np.zeros((S_, G, nb), dtype=np.float32),
               kc=np.zeros((S_, G, Nc, dk)), vc=np.zeros((S_, G, Nc, dv)))
    for si, b in enumerate(seqs):
        Tb = lens[b]
        assert 1 <= Tb <= T, "a sequence holds between 1 and T tokens"
        Ncb = num_compressed(Tb, params.l, params.d)
        nbb = -(-Tb // params.lsel)
        t_rows = np.array([Tb - 1])
        qb = to_f64(q_t[b])
        gb = to_f64(inp["gates"][b])
        for g in range(G):
            K = to_f64(kcache[b, g, :Tb])
            V = to_f64(vcache[b, g, :Tb])
            Kc = compress(K, pe_k, w_k, params.l, params.d) if kc is None else kc[b, g, :Ncb]
            Vc = compress(V, pe_v, w_v, params.l, params.d) if vc is None else vc[b, g, :Ncb]
            res["kc"][si, g, :Ncb], res["vc"][si, g, :Ncb] = Kc, Vc
            hs = slice(g * hpg, (g + 1) * hpg)
            r = nsa_group_rows(qb[None, hs], t_rows, K, V, Kc, Vc, gb[None, hs], params, scale)
            for key in ("out", "o_cmp", "o_slc", "o_win"):
                res[key][si, hs] = r[key][0]
            res["idx"][si, g] = r["idx"][0]
            res["S"][si, g, :nbb] = r["S"][0]
            res["S32"][si, g, :nbb] = r["S32"][0]
    res["seqs"] = np.array(seqs)
    res["lens"] = np.array([lens[b] for b in seqs])
    return res


def nsa_decode_multi_reference(inp: Dict[str, torch.Tensor], seqs: Optional[Iterable[int]] = None,
                               params: NSAParams = NSAParams(),
                               kc: Optional[np.ndarray] = None, vc: Optional[np.ndarray] = None
                               ) -> Dict[str, np.ndarray]:
    """Decode of m query tokens per sequence at positions T-m .. T-1 (all in
    the caches): rows T-m .. T-1 of the same definition, each with its own
    selection (several draft tokens checked at once, or a short chunk).

    inp: ``workloads.make_decode_multi`` (caches [B,G,T,d], q [B,m,H,dk],
    gates [B,m,H,3]).  kc/vc: optional compressed caches [B,G,Nc,d] (fp64);
    computed here when absent.  Returns out [S,m,H,dv], o_cmp/o_slc/o_win,
    idx [S,m,G,n] and S32 [S,m,G,nb].
    """
    kcache, vcache, q_t = inp["kcache"], inp["vcache"], inp["q"]
    B, G, T, dk = kcache.shape
    m, H = q_t.shape[1], q_t.shape[2]
    dv = vcache.shape[3]
    hpg = H // G
    scale = 1.0 / math.sqrt(dk)
    seqs = list(range(B)) if seqs is None else list(seqs)
    pe_k, pe_v = to_f64(inp["pe_k"]), to_f64(inp["pe_v"])
    w_k, w_v = to_f64(inp["w_k"]), to_f64(inp["w_v"])
    nb = -(-T // params.lsel)
    res = dict(out=np.zeros((len(seqs), m, H, dv)), o_cmp=np.zeros((len(seqs), m, H, dv)),
               o_slc=np.zeros((len(seqs), m, H, dv)), o_win=np.zeros((len(seqs), m, H, dv)),
               idx=np.zeros((len(seqs), m, G, params.n), dtype=np.int32),
               S32=np.zeros((len(seqs), m, G, nb), dtype=np.float32))
    t_rows = np.arange(T - m, T)
    for si, b in enumerate(seqs):
        qb = to_f64(q_t[b])
        gb = to_f64(inp["gates"][b])
        for g in range(G):
            K = to_f64(kcache[b, g])
            V = to_f64(vcache[b, g])
            Kc = compress(K, pe_k, w_k, params.l, params.d) if kc is None else kc[b, g]
            Vc = compress(V, pe_v, w_v, params.l, params.d) if vc is None else vc[b, g]
            hs = slice(g * hpg, (g + 1) * hpg)
            r = nsa_group_rows(qb[:, hs], t_rows, K, V, Kc, Vc, gb[:, hs], params, scale)
            for key in ("out", "o_cmp", "o_slc", "o_win"):
                res[key][si, :, hs] = r[key]
            res["idx"][si, :, g] = r["idx"]
            res["S32"][si, :, g] = r["S32"]
    res["seqs"] = np.array(seqs)
    return res


def decode_tokens_read(T: int, params: NSAParams = NSAParams()) -> Dict[str, int]:
    """Positions one decode step reads per KV head at context T (query t=T-1).

    compressed = |C_{T-1}|, selected = tokens of the n kept blocks (all
    causal), window = min(w, T).  The pages' own accounting at 64k [P2 III.3]
    uses T/d compressed tokens: 4096 + 16*64 + 512 = 5632.
    """
    Nc = num_compressed(T, params.l, params.d)
    ncmp = int(num_visible_compressed(T - 1, params.l, params.d, Nc))
    jt = (T - 1) // params.lsel
    nsel_blocks = min(params.n, jt + 1)
    # every kept block is complete except possibly the query's own block j_t
    sel = (nsel_blocks - 1) * params.lsel + (T - jt * params.lsel)
    return dict(compressed=ncmp, selected=sel, window=min(params.w, T))
