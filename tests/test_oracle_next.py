"""Pins of the oracles written ahead of their kernels (the next rows of the
hot-path scope): DSA prefill (every position a query).  CPU only."""
import math

import numpy as np

from oracle import dsa as D
from oracle import nsa as O
from workloads import DSAWorkload, make_dsa_prefill

DSA_SMALL = DSAWorkload("dsa_prefill_T300_HI2_dI16_H4_dk32_dv24_top64", 1, 300, 2, 16, 4, 32, 24, 64, 9)


def test_dsa_prefill_full_causal_attention_when_topk_covers_the_prefix():
    """topk >= t + 1 keeps every causal position: each row is textbook causal
    softmax attention."""
    inp = make_dsa_prefill(DSA_SMALL, T=120)
    rows = [0, 1, 37, 119]
    got = D.dsa_prefill_reference(inp, topk=1000, rows=rows)["out"]
    q, K, V = O.to_f64(inp["q"][0]), O.to_f64(inp["k"][0]), O.to_f64(inp["v"][0])
    scale = 1.0 / math.sqrt(q.shape[-1])
    for r, t in enumerate(rows):
        z = (q[t] @ K[: t + 1].T) * scale
        p = np.exp(z - z.max(axis=1, keepdims=True))
        p /= p.sum(axis=1, keepdims=True)
        np.testing.assert_allclose(got[r], p @ V[: t + 1], rtol=1e-12, atol=1e-12)


def test_dsa_prefill_last_row_is_the_decode_step():
    """Row T-1 of the prefill is the decode step whose query is that row."""
    inp = make_dsa_prefill(DSA_SMALL)
    T = DSA_SMALL.T
    pre = D.dsa_prefill_reference(inp, DSA_SMALL.topk, rows=[T - 1])
    dec_inp = dict(qI=inp["qI"][:, T - 1], wI=inp["wI"][:, T - 1], kI=inp["kI"], q=inp["q"][:, T - 1],
                   k=inp["k"], v=inp["v"])
    dec = D.dsa_decode_reference(dec_inp, DSA_SMALL.topk)
    np.testing.assert_array_equal(pre["idx"][0], dec["idx"][0])
    np.testing.assert_allclose(pre["out"][0], dec["out"][0], rtol=1e-13, atol=1e-13)


def test_dsa_prefill_selection_brute_force():
    """Scores by explicit loops, selection by sorting (-score, position)
    tuples: the kept set of every sampled row, and nothing after t."""
    inp = make_dsa_prefill(DSA_SMALL)
    qI, wI, kI = (O.to_f64(inp[n][0]) for n in ("qI", "wI", "kI"))
    rows = [5, 63, 64, 150, 299]
    res = D.dsa_prefill_reference(inp, DSA_SMALL.topk, rows=rows)
    for r, t in enumerate(rows):
        scores = []
        for s in range(t + 1):
            acc = 0.0
            for h in range(qI.shape[1]):
                acc += wI[t, h] * max(0.0, sum(qI[t, h, e] * kI[s, e] for e in range(qI.shape[2])))
            scores.append((-float(np.float32(acc)), s))
        keep = sorted(s for _, s in sorted(scores)[: min(DSA_SMALL.topk, t + 1)])
        assert res["idx"][r].tolist() == keep, t
        assert res["idx"][r].max() <= t


# ---------------------------------------------------------------- multi-token decode
import torch  # noqa: E402

from workloads import DecodeWorkload, NSAParams, make_decode, make_decode_multi  # noqa: E402

DEC_SMALL = DecodeWorkload("nsa_decode_B2_T1500_H4_G2_d32", 2, 1500, 4, 2, 32, 32, 13)


def test_multi_token_decode_with_one_token_is_the_decode_step():
    one = make_decode_multi(DEC_SMALL, 1)
    ref = make_decode(DEC_SMALL)
    assert torch.equal(one["q"][:, 0], ref["q"]) and torch.equal(one["gates"][:, 0], ref["gates"])
    got = O.nsa_decode_multi_reference(one)
    dec = O.nsa_decode_reference(ref)
    np.testing.assert_array_equal(got["idx"][:, 0], dec["idx"])
    np.testing.assert_allclose(got["out"][:, 0], dec["out"], rtol=0, atol=0)


def test_multi_token_decode_rows_are_the_prefill_rows():
    """Token-major copies of the caches and the m queries placed at rows
    T-m .. T-1 of a prefill input give the same rows."""
    m, T = 5, DEC_SMALL.T
    inp = make_decode_multi(DEC_SMALL, m)
    got = O.nsa_decode_multi_reference(inp, seqs=[1])
    b = 1
    q = torch.zeros(1, T, DEC_SMALL.H, DEC_SMALL.dk, dtype=torch.bfloat16)
    q[0, T - m:] = inp["q"][b]
    gates = torch.zeros(1, T, DEC_SMALL.H, 3, dtype=torch.bfloat16)
    gates[0, T - m:] = inp["gates"][b]
    pre_inp = dict(q=q, k=inp["kcache"][b].transpose(0, 1)[None], v=inp["vcache"][b].transpose(0, 1)[None],
                   pe_k=inp["pe_k"], pe_v=inp["pe_v"], w_k=inp["w_k"], w_v=inp["w_v"], gates=gates)
    pre = O.nsa_prefill_reference(pre_inp, rows=range(T - m, T))
    np.testing.assert_array_equal(got["idx"][0], pre["idx"])
    np.testing.assert_allclose(got["out"][0], pre["out"], rtol=0, atol=0)
    jt = (T - 1) // NSAParams().lsel
    for r in range(m):                               # forced blocks of every token
        t = T - m + r
        for g in range(DEC_SMALL.G):
            assert {0, t // 64 - 1, t // 64} <= set(got["idx"][0, r, g].tolist())
    assert jt >= NSAParams().n                       # a real top-n choice is made
