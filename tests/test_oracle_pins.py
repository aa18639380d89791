"""Pins of the fp64 oracle against facts that do not come from the oracle itself:
numbers the pages print (tests/golden/page_facts.json), closed forms, textbook
or library routines (torch SDPA / matmul / unfold), brute force on tiny inputs
and invariants.  CPU only."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import nsa as O
from oracle import dsa as D
from workloads import NSAParams, PREFILL_CONFIGS, make_prefill, make_dsa, dsa_config


def _facts(golden_dir):
    with open(os.path.join(golden_dir, "page_facts.json")) as f:
        return json.load(f)


# ----------------------------------------------------------------- page facts
def test_hyper_parameters_match_pages(golden_dir):
    f = _facts(golden_dir)["nsa_hyper_parameters"]
    p = NSAParams()
    assert (p.l, p.d, p.lsel, p.n, p.w) == (f["l"], f["d"], f["lsel"], f["n"], f["w"])
    assert f["forced_initial"] + f["forced_local"] == 3


def test_decode_token_accounting_64k(golden_dir):
    f = _facts(golden_dir)["decode_tokens_64k"]
    p = NSAParams()
    T = f["context"]
    # the pages' accounting: T/d compressed + n*l' selected + w window
    assert T // p.d + p.n * p.lsel + p.w == f["nsa_tokens"]
    assert T == f["full_tokens"]
    # the exact count of complete compression windows is one less (16i+32 <= T)
    r = O.decode_tokens_read(T, p)
    assert r == dict(compressed=4095, selected=1024, window=512)
    assert r["compressed"] + r["selected"] + r["window"] == f["nsa_tokens"] - 1


def test_dsa_fraction(golden_dir):
    f = _facts(golden_dir)["dsa_selection"]
    assert f["context"] // f["topk"] == f["ops_ratio"]
    assert round(100.0 * f["topk"] / f["context"], 1) == f["percent_rounded"]
    wl = dsa_config()
    assert (wl.T, wl.topk) == (f["context"], f["topk"])


# ----------------------------------------------------------------- bf16 rounding
def test_bf16_round_matches_torch_on_fp32_inputs():
    g = torch.Generator().manual_seed(123)
    x32 = torch.randn(200000, generator=g) * torch.exp(torch.randn(200000, generator=g) * 8)
    ref = x32.to(torch.bfloat16).to(torch.float64).numpy()
    got = O.bf16_round(x32.to(torch.float64).numpy())
    np.testing.assert_array_equal(got, ref)


def test_bf16_round_ties_to_even():
    one = 1.0
    ulp = 2.0 ** -7
    assert O.bf16_round(np.array([one + ulp / 2]))[0] == one            # tie -> even (1.0)
    assert O.bf16_round(np.array([one + 3 * ulp / 2]))[0] == one + 2 * ulp
    assert O.bf16_round(np.array([one + ulp / 2 + 1e-12]))[0] == one + ulp
    assert O.bf16_round(np.array([-(one + ulp / 2)]))[0] == -one
    assert O.bf16_round(np.array([0.0]))[0] == 0.0


# ----------------------------------------------------------------- compression
@pytest.mark.parametrize("T,expect", [(65536, 4095), (8192, 511), (2048, 127), (31, 0), (32, 1),
                                      (47, 1), (48, 2), (1000, 61)])
def test_num_compressed(T, expect):
    assert O.num_compressed(T, 32, 16) == expect


def test_compress_mean_pool_closed_form():
    # W = stacked I/l and PE = 0 turn phi into the block mean
    rng = np.random.default_rng(0)
    T, dX, l, d = 200, 8, 32, 16
    X = O.bf16_round(rng.standard_normal((T, dX)))
    W = np.concatenate([np.eye(dX) / l for _ in range(l)], axis=0)
    got = O.compress(X, np.zeros((l, dX)), W, l, d)
    csum = np.concatenate([np.zeros((1, dX)), np.cumsum(X, axis=0)])
    Nc = (T - l) // d + 1
    starts = d * np.arange(Nc)
    mean = (csum[starts + l] - csum[starts]) / l
    np.testing.assert_allclose(got, O.bf16_round(mean), rtol=0, atol=0)


def test_compress_matches_torch_unfold_matmul():
    rng = np.random.default_rng(1)
    T, dX, dout, l, d = 333, 16, 24, 32, 16
    X = O.bf16_round(rng.standard_normal((T, dX)))
    PE = O.bf16_round(0.02 * rng.standard_normal((l, dX)))
    W = O.bf16_round(rng.standard_normal((l * dX, dout)) / math.sqrt(l * dX))
    got = O.compress(X, PE, W, l, d)
    xt = torch.from_numpy(X)
    win = xt.unfold(0, l, d)                       # [Nc, dX, l]
    win = win.permute(0, 2, 1) + torch.from_numpy(PE)
    ref = torch.matmul(win.reshape(win.shape[0], -1), torch.from_numpy(W)).numpy()
    assert got.shape == ref.shape == ((T - l) // d + 1, dout)
    np.testing.assert_array_equal(got, O.bf16_round(ref))


# ----------------------------------------------------------------- compressed attention
def _sdpa(q, K, V, causal=False, scale=None):
    """torch SDPA in fp64 on CPU: q [R,dk], K [S,dk], V [S,dv]."""
    qt = torch.from_numpy(q)[None, None]
    kt = torch.from_numpy(K)[None, None]
    vt = torch.from_numpy(V)[None, None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=causal, scale=scale)
    return o[0, 0].numpy()


def test_cmp_attention_all_visible_is_textbook_attention():
    rng = np.random.default_rng(2)
    Nc, dk, dv, l, d = 20, 16, 8, 32, 16
    Kc, Vc = rng.standard_normal((Nc, dk)), rng.standard_normal((Nc, dv))
    t = np.array([d * (Nc - 1) + l - 1, 5000])           # both see every block
    q = rng.standard_normal((2, 3, dk))
    o, p = O.cmp_attention(q, t, Kc, Vc, 1 / math.sqrt(dk), l, d)
    for r in range(2):
        np.testing.assert_allclose(o[r], _sdpa(q[r], Kc, Vc), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(p.sum(-1), 1.0, rtol=1e-12)


def test_cmp_attention_causality_and_empty():
    rng = np.random.default_rng(3)
    Nc, dk, dv, l, d = 12, 8, 8, 32, 16
    Kc, Vc = rng.standard_normal((Nc, dk)), rng.standard_normal((Nc, dv))
    t = np.array([0, 30, 31, 46, 47, 100])
    q = rng.standard_normal((t.size, 2, dk))
    o, p = O.cmp_attention(q, t, Kc, Vc, 0.3, l, d)
    nvis = O.num_visible_compressed(t, l, d, Nc)
    assert nvis.tolist() == [0, 0, 1, 1, 2, 5]
    assert np.all(o[:2] == 0) and np.all(p[:2] == 0)
    # t=31 sees exactly block 0 -> output is Vc[0]
    np.testing.assert_allclose(o[2], np.broadcast_to(Vc[0], (2, dv)), rtol=1e-14)
    # changing invisible blocks changes nothing
    Kc2, Vc2 = Kc.copy(), Vc.copy()
    Kc2[5:] += 10.0
    Vc2[5:] -= 3.0
    o2, _ = O.cmp_attention(q, t, Kc2, Vc2, 0.3, l, d)
    np.testing.assert_array_equal(o, o2)


def test_cmp_attention_no_complete_block():
    # T < l: no compressed block exists, the branch output is 0
    rng = np.random.default_rng(5)
    o, p = O.cmp_attention(rng.standard_normal((3, 2, 8)), np.array([0, 10, 30]), np.zeros((0, 8)),
                           np.zeros((0, 4)), 0.3, 32, 16)
    assert o.shape == (3, 2, 4) and np.all(o == 0) and p.shape == (3, 2, 0)


# ----------------------------------------------------------------- block scores
def test_overlap_matrix_brute_force():
    l, d, lsel = 32, 16, 64
    Nc, nb = 40, 12
    Om = O.overlap_matrix(Nc, nb, l, d, lsel)
    for i in range(Nc):
        a = set(range(d * i, d * i + l))
        for j in range(nb):
            b = set(range(lsel * j, lsel * j + lsel))
            assert Om[i, j] * d == len(a & b)
    # chunk counts 1,2,2,2,1 for i = 4j-1 .. 4j+3
    assert Om[3:8, 1].tolist() == [1, 2, 2, 2, 1]


def test_block_scores_one_hot_and_conservation():
    l, d, lsel = 32, 16, 64
    Nc, nb = 30, 9
    p = np.zeros((1, 2, Nc))
    p[0, 0, 7] = 1.0            # head 0 puts all mass on compressed block 7 (tokens 112..143)
    p[0, 1, 8] = 1.0            # head 1 on block 8 (tokens 128..159)
    S = O.block_scores(p, nb, l, d, lsel)[0]
    expect = np.zeros(nb)
    expect[1] = 1.0             # block 7 shares chunk 7 (112..127) with selection block 1
    expect[2] = 1.0 + 2.0       # chunk 8 of block 7; chunks 8, 9 of block 8
    np.testing.assert_array_equal(S, expect)
    # conservation: each visible compressed block spreads l/d chunks
    rng = np.random.default_rng(4)
    logits = rng.standard_normal((5, 16, Nc))
    pr = np.exp(logits) / np.exp(logits).sum(-1, keepdims=True)
    S = O.block_scores(pr, nb, l, d, lsel)
    np.testing.assert_allclose(S.sum(-1), (l / d) * 16, rtol=1e-12)


# ----------------------------------------------------------------- top-n selection
def _brute_select(S32, t, n, lsel):
    jt = t // lsel
    if jt + 1 <= n:
        return sorted(range(jt + 1)) + [-1] * (n - jt - 1)
    forced = sorted({0, jt, jt - 1})
    rest = sorted((j for j in range(jt + 1) if j not in forced),
                  key=lambda j: (-float(S32[j]), j))
    return sorted(forced + rest[: n - len(forced)])


@pytest.mark.parametrize("seed", range(6))
def test_select_blocks_brute_force(seed):
    rng = np.random.default_rng(seed)
    n, lsel = 16, 64
    for _ in range(40):
        t = int(rng.integers(0, 4000))
        nb = t // lsel + 1
        if seed % 2:
            S = rng.integers(0, 4, size=nb).astype(np.float32)   # many exact ties
        else:
            S = rng.random(nb).astype(np.float32)
        got = O.select_blocks(S, t, n, lsel).tolist()
        assert got == _brute_select(S, t, n, lsel)
        jt = t // lsel
        kept = [j for j in got if j >= 0]
        assert len(kept) == min(n, jt + 1) == len(set(kept))
        assert all(0 <= j <= jt for j in kept)
        assert {0, jt, max(jt - 1, 0)} <= set(kept)
        assert kept == sorted(kept)


def test_selection_alternatives_band():
    # t in block 7, n=4: forced {0, 6, 7}; one free pick among {1..5}; blocks 1 and 2 nearly tie
    S = np.array([5, 0.5000001, 0.5, 0.3, 0.2, 0.1, 9, 9], dtype=np.float32)
    gap, definite, band, need = O.selection_alternatives(S, 7 * 64, 4, 64, 1e-5)
    assert 0 < gap < 1e-5
    assert definite == {0, 6, 7} and band == {1, 2} and need == 1
    assert O.select_blocks(S, 7 * 64, 4, 64).tolist() == [0, 1, 6, 7]
    # a clear winner leaves no band
    S[1] = 0.9
    gap, definite, band, need = O.selection_alternatives(S, 7 * 64, 4, 64, 1e-5)
    assert gap > 0.1 and definite == {0, 1, 6, 7} and band == set() and need == 0


# ----------------------------------------------------------------- full-attention reductions
def _small_inputs(T, seed=0):
    wl = PREFILL_CONFIGS["tiny_2k"]
    inp = make_prefill(wl, T=T)
    return wl, inp


def _full_causal(inp, g_rows=None):
    q = O.to_f64(inp["q"][0])            # [T,H,dk]
    k = O.to_f64(inp["k"][0])            # [T,G,dk]
    v = O.to_f64(inp["v"][0])
    T, H, dk = q.shape
    G = k.shape[1]
    out = np.zeros((T, H, v.shape[2]))
    for h in range(H):
        g = h // (H // G)
        out[:, h] = _sdpa(q[:, h], k[:, g], v[:, g], causal=True)
    return out


def test_selection_only_equals_full_attention_when_all_blocks_fit():
    T = 1000                              # n*l' = 1024 >= T: every block is selected
    wl, inp = _small_inputs(T)
    inp["gates"] = torch.zeros_like(inp["gates"])
    inp["gates"][..., 1] = 1.0
    res = O.nsa_prefill_reference(inp)
    np.testing.assert_allclose(res["out"], _full_causal(inp), rtol=0, atol=1e-12)


def test_window_only_equals_full_attention_when_window_covers_sequence():
    T = 700
    wl, inp = _small_inputs(T)
    inp["gates"] = torch.zeros_like(inp["gates"])
    inp["gates"][..., 2] = 1.0
    res = O.nsa_prefill_reference(inp, params=NSAParams(w=T))
    np.testing.assert_allclose(res["out"], _full_causal(inp), rtol=0, atol=1e-12)


def test_window_rows_before_w_are_full_attention():
    T = 1300
    wl, inp = _small_inputs(T)
    rows = [0, 1, 100, 511, 512, 1299]
    res = O.nsa_prefill_reference(inp, rows=rows)
    full = _full_causal(inp)
    for r, t in enumerate(rows):
        if t < 512:
            np.testing.assert_allclose(res["o_win"][r], full[t], rtol=0, atol=1e-12)
        else:
            assert np.abs(res["o_win"][r] - full[t]).max() > 1e-6


def test_uniform_attention_gives_plain_means():
    # K = 0 makes every logit equal: each branch is then the plain mean of V over its key set
    T = 1500
    wl, inp = _small_inputs(T)
    inp["k"] = torch.zeros_like(inp["k"])
    rows = [0, 5, 511, 512, 513, 1023, 1024, 1499]
    res = O.nsa_prefill_reference(inp, rows=rows)
    V = O.to_f64(inp["v"][0, :, 0])                      # G = 1
    csum = np.concatenate([np.zeros((1, V.shape[1])), np.cumsum(V, axis=0)])
    for r, t in enumerate(rows):
        lo = max(0, t - 512 + 1)
        win_mean = (csum[t + 1] - csum[lo]) / (t + 1 - lo)
        np.testing.assert_allclose(res["o_win"][r], np.broadcast_to(win_mean, res["o_win"][r].shape),
                                   rtol=0, atol=1e-12)
        keys = [s for j in res["idx"][r, 0] if j >= 0 for s in range(64 * j, min(64 * j + 64, t + 1))]
        np.testing.assert_allclose(res["o_slc"][r], np.broadcast_to(V[keys].mean(0), res["o_slc"][r].shape),
                                   rtol=0, atol=1e-12)


def test_prefill_invariants_tiny_config():
    T = 2048
    wl, inp = _small_inputs(T)
    rows = list(range(0, T, 37)) + [T - 1]
    res = O.nsa_prefill_reference(inp, rows=rows)
    hpg = wl.H // wl.G
    for r, t in enumerate(rows):
        for g in range(wl.G):
            kept = [j for j in res["idx"][r, g] if j >= 0]
            jt = t // 64
            assert len(kept) == min(16, jt + 1)
            assert {0, jt, max(jt - 1, 0)} <= set(kept)
            if t >= 31:
                np.testing.assert_allclose(res["S"][r, g].sum(), 2.0 * hpg, rtol=1e-12)
    # gates combine linearly
    gates = O.to_f64(inp["gates"][0, rows])
    comb = (gates[..., 0:1] * res["o_cmp"] + gates[..., 1:2] * res["o_slc"]
            + gates[..., 2:3] * res["o_win"])
    np.testing.assert_allclose(res["out"], comb, rtol=1e-14)


def test_decode_equals_last_prefill_row():
    T = 1500
    wl, inp = _small_inputs(T)
    pre = O.nsa_prefill_reference(inp, rows=[T - 1])
    dec_inp = dict(kcache=inp["k"].permute(0, 2, 1, 3).contiguous(),
                   vcache=inp["v"].permute(0, 2, 1, 3).contiguous(),
                   q=inp["q"][:, T - 1], gates=inp["gates"][:, T - 1],
                   pe_k=inp["pe_k"], pe_v=inp["pe_v"], w_k=inp["w_k"], w_v=inp["w_v"])
    dec = O.nsa_decode_reference(dec_inp)
    np.testing.assert_array_equal(dec["idx"][0], pre["idx"][0])
    np.testing.assert_allclose(dec["out"][0], pre["out"][0], rtol=0, atol=1e-13)


# ----------------------------------------------------------------- DSA
def test_decode_with_lengths_equals_cropped_caches():
    """A sequence of length L inside a larger cache is decoded exactly as the
    same L tokens alone: nothing past L is read."""
    from workloads import decode_config, make_decode
    wl = decode_config()
    inp = make_decode(wl, B=3, T=700)
    lens = [700, 64, 333]
    res = O.nsa_decode_reference(inp, seq_lens=lens)
    for b, L in enumerate(lens):
        one = {k: v for k, v in inp.items()}
        for key in ("kcache", "vcache"):
            big = inp[key][b:b + 1, :, :L].clone()
            one[key] = big
        for key in ("q", "gates"):
            one[key] = inp[key][b:b + 1]
        ref = O.nsa_decode_reference(one)
        np.testing.assert_array_equal(res["out"][b], ref["out"][0])
        np.testing.assert_array_equal(res["idx"][b], ref["idx"][0])
    # poisoning the rows past each length changes nothing
    for key in ("kcache", "vcache"):
        for b, L in enumerate(lens):
            inp[key][b, :, L:] = 1e4
    res2 = O.nsa_decode_reference(inp, seq_lens=lens)
    np.testing.assert_array_equal(res["out"], res2["out"])


def test_dsa_indexer_brute_force():
    rng = np.random.default_rng(7)
    HI, dI, T = 3, 5, 40
    qI, wI, kI = rng.standard_normal((HI, dI)), rng.standard_normal(HI), rng.standard_normal((T, dI))
    got = D.dsa_indexer_scores(qI, wI, kI)
    for s in range(T):
        acc = 0.0
        for h in range(HI):
            dot = sum(qI[h, c] * kI[s, c] for c in range(dI))
            acc += wI[h] * (dot if dot > 0 else 0.0)
        assert abs(got[s] - acc) < 1e-12
    # ReLU: a key anti-aligned with every indexer head scores exactly 0
    kI2 = -np.abs(kI)
    assert np.all(D.dsa_indexer_scores(np.abs(qI), wI, kI2) == 0)


@pytest.mark.parametrize("seed", range(4))
def test_dsa_topk_brute_force(seed):
    rng = np.random.default_rng(seed)
    T, k = 300, 37
    I = (rng.integers(-3, 4, size=T) if seed % 2 else rng.standard_normal(T)).astype(np.float32)
    got = D.topk_positions(I, k).tolist()
    ref = sorted(sorted(range(T), key=lambda s: (-float(I[s]), s))[:k])
    assert got == ref
    assert D.topk_positions(I, T + 5).tolist() == list(range(T))


# ----------------------------------------------------------------- acceptance of differing top-k sets
def _brute_acceptable(scores, k):
    """Every k-subset that a ranking consistent with the scores can produce:
    no dropped position scores strictly above a kept one (exact ties free)."""
    import itertools
    T = len(scores)
    out = set()
    for X in itertools.combinations(range(T), k):
        xs = set(X)
        lo = min(float(scores[x]) for x in X)
        hi = max((float(scores[y]) for y in range(T) if y not in xs), default=-np.inf)
        if lo >= hi:
            out.add(X)
    return out


@pytest.mark.parametrize("seed", range(6))
def test_topk_set_valid_brute_force(seed):
    # integer-valued scores (exact ties) far apart relative to the tolerance:
    # the sets the predicate accepts are exactly the tie-permuted top-k sets
    import itertools
    rng = np.random.default_rng(100 + seed)
    T, k = 9, 4
    I = (rng.integers(0, 4, size=T) * 10 + 50).astype(np.float32)
    acc = {X for X in itertools.combinations(range(T), k) if D.topk_set_valid(I, X, k, 1e-5)[0]}
    assert acc == _brute_acceptable(I, k)
    assert tuple(D.topk_positions(I, k).tolist()) in acc


def test_topk_alternatives_cases():
    # an exact tie at the cut: both tied positions in the band, one of them needed
    I = np.array([9, 5, 7, 5, 1, 0], dtype=np.float32)
    gap, above, band, need = D.topk_alternatives(I, 3, 1e-5)
    assert gap == 0 and set(above.tolist()) == {0, 2} and set(band.tolist()) == {1, 3} and need == 1
    assert D.topk_positions(I, 3).tolist() == [0, 1, 2]          # the tie goes to the lower position
    assert D.topk_set_valid(I, [0, 2, 3], 3, 1e-5)[0]            # the other side of the tie is acceptable
    # a clear gap: empty band, nothing needed
    gap, above, band, need = D.topk_alternatives(I, 2, 1e-5)
    assert gap > 0.1 and set(above.tolist()) == {0, 2} and band.size == 0 and need == 0
    # k >= T keeps everything
    gap, above, band, need = D.topk_alternatives(I, 6, 1e-5)
    assert gap == float("inf") and above.tolist() == list(range(6)) and need == 0
    assert D.topk_set_valid(I, range(6), 9, 1e-5)[0]
    # a near-tie inside the tolerance is a band, one outside is not
    J = np.array([3.0, 2.0, 2.0 * (1 + 4e-6), 1.0], dtype=np.float32)
    assert set(D.topk_alternatives(J, 2, 1e-5)[2].tolist()) == {1, 2}
    assert D.topk_alternatives(J, 2, 1e-7)[2].size == 0


def test_topk_set_valid_rejects_planted_invalid_sets():
    I = np.array([9, 5, 7, 5, 1, 0], dtype=np.float32)
    ok = lambda X, k=3: D.topk_set_valid(I, X, k, 1e-5)[0]
    assert ok([0, 1, 2]) and ok([2, 0, 3])
    assert not ok([0, 1, 3])              # drops position 2, clearly above the cut
    assert not ok([0, 2, 4])              # takes position 4, below the band
    assert not ok([0, 2])                 # too few
    assert not ok([0, 2, 1, 3])           # too many
    assert not ok([0, 2, 2])              # a duplicate
    assert not ok([0, 2, 6])              # out of range
    assert not ok([0, 1, 2], k=4)         # k=4 needs 4 positions


@pytest.mark.parametrize("seed", range(4))
def test_selection_set_valid_brute_force(seed):
    # NSA rows: forced blocks {0, j_t-1, j_t}; integer scores with exact ties
    import itertools
    rng = np.random.default_rng(200 + seed)
    n, lsel = 6, 64
    jt = 9
    t = jt * lsel + 5
    S = (rng.integers(0, 3, size=jt + 1) * 4 + 1).astype(np.float32)
    forced = {0, jt - 1, jt}
    free = [j for j in range(jt + 1) if j not in forced]
    brute = {tuple(sorted(forced | {free[i] for i in X})) for X in _brute_acceptable(S[free], n - 3)}
    acc = set()
    for X in itertools.combinations(free, n - 3):
        row = sorted(forced | set(X))
        if O.selection_set_valid(S, t, row, n, lsel, 1e-5)[0]:
            acc.add(tuple(row))
    assert acc == brute
    assert tuple(O.select_blocks(S, t, n, lsel).tolist()) in acc


def test_selection_set_valid_rejects_planted_invalid_rows():
    S = np.array([5, 0.5000001, 0.5, 0.3, 0.2, 0.1, 9, 9], dtype=np.float32)
    t, n, lsel = 7 * 64, 4, 64
    ok = lambda row: O.selection_set_valid(S, t, row, n, lsel, 1e-5)[0]
    assert ok([0, 1, 6, 7]) and ok([0, 2, 6, 7])      # the near-tie resolves either way
    assert not ok([0, 3, 6, 7])                        # below the band
    assert not ok([1, 2, 6, 7])                        # drops forced block 0
    assert not ok([0, 1, 5, 7])                        # drops forced block j_t - 1
    assert not ok([0, 6, 1, 7])                        # not ascending
    assert not ok([0, 1, 1, 7])                        # duplicate
    # a short row (j_t + 1 <= n) keeps every block and pads with -1
    assert O.selection_set_valid(S, 2 * 64, [0, 1, 2, -1], n, lsel, 1e-5)[0]
    assert not O.selection_set_valid(S, 2 * 64, [0, 1, -1, 2], n, lsel, 1e-5)[0]
    assert not O.selection_set_valid(S, 2 * 64, [0, 2, -1, -1], n, lsel, 1e-5)[0]


def test_dsa_with_lengths_equals_cropped_context():
    """A row whose context holds T_b tokens is the same step on the first T_b
    tokens alone; nothing past T_b is read."""
    wl = dsa_config()
    inp = make_dsa(wl, B=3, T=900)
    lens = [900, 37, 512]
    res = D.dsa_decode_reference(inp, topk=64, seq_lens=lens)
    for b, L in enumerate(lens):
        one = {key: (t[b:b + 1, :L] if key in ("kI", "k", "v") else t[b:b + 1]) for key, t in inp.items()}
        ref = D.dsa_decode_reference(one, topk=64)
        np.testing.assert_array_equal(res["out"][b], ref["out"][0])
        kk = min(64, L)
        np.testing.assert_array_equal(res["idx"][b, :kk], ref["idx"][0])
        assert (res["idx"][b, kk:] == -1).all()
    for key in ("kI", "k", "v"):
        for b, L in enumerate(lens):
            inp[key][b, L:] = 50.0
    res2 = D.dsa_decode_reference(inp, topk=64, seq_lens=lens)
    np.testing.assert_array_equal(res["out"], res2["out"])


def test_dsa_full_when_k_covers_context():
    wl = dsa_config()
    inp = make_dsa(wl, B=2, T=300)
    res = D.dsa_decode_reference(inp, topk=512)
    for b in range(2):
        q = O.to_f64(inp["q"][b])
        K = O.to_f64(inp["k"][b])
        V = O.to_f64(inp["v"][b])
        ref = np.stack([_sdpa(q[h:h + 1], K, V)[0] for h in range(q.shape[0])])
        np.testing.assert_allclose(res["out"][b], ref, rtol=0, atol=1e-12)


def test_dsa_latent_values_when_k_covers_context():
    """Latent KV (values = first dv columns of the key rows): with top-k
    covering the context the step is full softmax attention over K with
    V = K[:, :dv]."""
    wl = dsa_config()
    inp = make_dsa(wl, B=2, T=300)
    inp["v"] = None
    res = D.dsa_decode_reference(inp, topk=512, latent_dv=wl.dv)
    assert res["out"].shape == (2, wl.H, wl.dv)
    for b in range(2):
        q = O.to_f64(inp["q"][b])
        K = O.to_f64(inp["k"][b])
        ref = np.stack([_sdpa(q[h:h + 1], K, K[:, :wl.dv])[0] for h in range(q.shape[0])])
        np.testing.assert_allclose(res["out"][b], ref, rtol=0, atol=1e-12)


def test_dsa_latent_values_need_dv_within_dk():
    wl = dsa_config()
    inp = make_dsa(wl, B=1, T=64)
    inp["v"] = None
    with pytest.raises(ValueError):
        D.dsa_decode_reference(inp, topk=8, latent_dv=wl.dk + 64)
