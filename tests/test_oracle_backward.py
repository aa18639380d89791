"""Pins of the NSA backward oracle (``oracle/nsa_bwd.py``), CPU only.

The backward is checked against things other than its own formulas: central
finite differences of the forward oracle (selection fixed, cache unrounded:
readings B1/B2), torch's automatic differentiation of an independent torch
formulation of the same forward, and closed forms.
"""
import math

import numpy as np
import pytest
import torch

from oracle import nsa as O
from oracle import nsa_bwd as BW
from workloads import NSAParams, PrefillWorkload, make_prefill, make_prefill_dout

# Rows of this case cover every regime: an empty compressed branch (t < 31),
# every block kept (j_t + 1 <= n), a real top-n choice (j_t >= n) and a
# window shorter than the context.
PARAMS = NSAParams(n=4, w=96)
WL = PrefillWorkload("nsa_bwd_T300_H4_G2_d16", 1, 300, 4, 2, 16, 16, 11, PARAMS)
GRADS = {"q": "dq", "k": "dk", "v": "dv", "gates": "dgates",
         "w_k": "dw_k", "w_v": "dw_v", "pe_k": "dpe_k", "pe_v": "dpe_v"}


def make_case():
    inp = make_prefill(WL)
    dout = O.to_f64(make_prefill_dout(WL)[0])
    idx = O.nsa_prefill_reference(inp, params=PARAMS)["idx"]
    return inp, dout, idx, BW._inputs_f64(inp, 0)


@pytest.fixture(scope="module")
def case():
    return make_case()


def _loss(x, dout, idx):
    return float((dout * BW.nsa_prefill_forward_fixed(x, idx, PARAMS)).sum())


def check_finite_differences(case):
    """<grad, U> against (f(x + eps U) - f(x - eps U)) / 2 eps for two seeded
    directions per input: one over every entry, one over the first 40 rows
    (or a random half of a parameter tensor)."""
    inp, dout, idx, x = case
    g = BW.nsa_prefill_backward(inp, dout, params=PARAMS, idx=idx, round_cache=False)
    rng = np.random.default_rng(5)
    eps = 1e-5
    for name, gname in GRADS.items():
        dirs = [rng.standard_normal(x[name].shape)]
        U2 = rng.standard_normal(x[name].shape)
        if name in ("q", "k", "v", "gates"):
            U2[40:] = 0.0
        else:
            U2 *= rng.random(x[name].shape) < 0.5
        dirs.append(U2)
        for U in dirs:
            xp = dict(x)
            xm = dict(x)
            xp[name] = x[name] + eps * U
            xm[name] = x[name] - eps * U
            fd = (_loss(xp, dout, idx) - _loss(xm, dout, idx)) / (2 * eps)
            an = float((g[gname] * U).sum())
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, fd, an)


def test_case_exercises_every_regime(case):
    _, _, idx, _ = case
    T = WL.T
    assert T - 1 >= PARAMS.n * PARAMS.lsel          # real top-n rows exist
    assert PARAMS.w < T and PARAMS.l - 1 > 0          # window shorter than the context; empty cmp rows
    jt = (T - 1) // PARAMS.lsel
    assert set(idx[T - 1, 0].tolist()) >= {0, jt - 1, jt}


def test_backward_matches_finite_differences(case):
    check_finite_differences(case)


def _torch_forward_loss(xt, dout, idx):
    """The forward written again in torch fp64 (kept blocks fixed, cache
    unrounded), for torch.autograd."""
    out = _torch_forward_out(xt, idx)
    return (torch.as_tensor(dout) * out).sum()


def _torch_forward_out(xt, idx, round_cache=False):
    """out [T, H, dv] of the forward written in torch fp64 from the
    definition: compression as flatten(X + PE) @ W (rounded to bf16 when
    ``round_cache``), then per query row softmax attention over the visible
    compressed entries, over the tokens of the kept blocks ``idx`` up to the
    row, and over the window, mixed by the gates (cmp, slc, win)."""
    q, k, v, gates = xt["q"], xt["k"], xt["v"], xt["gates"]
    T, H, dk = q.shape
    G, hpg = k.shape[1], H // k.shape[1]
    l, d, lsel, w = PARAMS.l, PARAMS.d, PARAMS.lsel, PARAMS.w
    scale = 1.0 / math.sqrt(dk)
    Nc = (T - l) // d + 1 if T >= l else 0

    def att(qs, Kk, Vk):
        return torch.softmax((qs @ Kk.T) * scale, dim=-1) @ Vk

    outs = []
    for g in range(G):
        K, V = k[:, g], v[:, g]
        Kc = torch.stack([(K[d * i: d * i + l] + xt["pe_k"]).reshape(-1) for i in range(Nc)]) @ xt["w_k"]
        Vc = torch.stack([(V[d * i: d * i + l] + xt["pe_v"]).reshape(-1) for i in range(Nc)]) @ xt["w_v"]
        if round_cache:
            Kc = Kc.to(torch.bfloat16).to(torch.float64)
            Vc = Vc.to(torch.bfloat16).to(torch.float64)
        rows = []
        hs = slice(g * hpg, (g + 1) * hpg)
        for t in range(T):
            qs = q[t, hs]
            nvis = min(Nc, (t - (l - 1)) // d + 1) if t >= l - 1 else 0
            o_c = att(qs, Kc[:nvis], Vc[:nvis]) if nvis else torch.zeros(hpg, V.shape[1], dtype=torch.float64)
            keys = [s for j in idx[t, g].tolist() if j >= 0 for s in range(j * lsel, min(j * lsel + lsel, t + 1))]
            keys = torch.as_tensor(keys, dtype=torch.long)
            o_s = att(qs, K[keys], V[keys])
            lo = max(0, t - w + 1)
            o_w = att(qs, K[lo:t + 1], V[lo:t + 1])
            gt = gates[t, hs]
            rows.append(gt[:, 0:1] * o_c + gt[:, 1:2] * o_s + gt[:, 2:3] * o_w)
        outs.append(torch.stack(rows))                  # [T, hpg, dv]
    return torch.cat(outs, dim=1)


def test_backward_matches_torch_autograd(case):
    inp, dout, idx, x = case
    g = BW.nsa_prefill_backward(inp, dout, params=PARAMS, idx=idx, round_cache=False)
    xt = {kk: torch.tensor(vv, dtype=torch.float64, requires_grad=True) for kk, vv in x.items()}
    _torch_forward_loss(xt, dout, idx).backward()
    for name, gname in GRADS.items():
        ref = xt[name].grad.numpy()
        np.testing.assert_allclose(g[gname], ref, rtol=1e-9, atol=1e-11, err_msg=name)


def test_single_key_closed_form():
    """One key: P = 1, O = V, so dS = dO.V - dO.O = 0: dq = 0, dK = 0, dV = dO."""
    rng = np.random.default_rng(1)
    q = rng.standard_normal((3, 8))
    K = rng.standard_normal((10, 8))
    V = rng.standard_normal((10, 5))
    dO = rng.standard_normal((3, 5))
    O_, dq, dK, dV = BW.attend_bwd(q, K, V, np.array([4]), 0.3, dO)
    np.testing.assert_allclose(O_, np.broadcast_to(V[4], (3, 5)), rtol=0, atol=1e-15)
    assert np.abs(dq).max() < 1e-14 and np.abs(dK).max() < 1e-14
    np.testing.assert_allclose(dV[0], dO.sum(axis=0), rtol=1e-14)


def test_zero_upstream_gradient(case):
    inp, _, idx, _ = case
    g = BW.nsa_prefill_backward(inp, np.zeros((WL.T, WL.H, WL.dv)), params=PARAMS, idx=idx)
    for gname in GRADS.values():
        assert not np.any(g[gname]), gname


def test_compress_backward_mean_pool_closed_form():
    """W = [I/l; ...; I/l] and PE = 0 make each compressed entry the mean of
    its l tokens, so token s receives sum over the blocks holding it of
    dXc_i / l, and PE row r receives sum_i dXc_i / l."""
    l, d, dx, T = 32, 16, 3, 100
    rng = np.random.default_rng(2)
    X = rng.standard_normal((T, dx))
    W = np.tile(np.eye(dx) / l, (l, 1))
    PE = np.zeros((l, dx))
    Nc = O.num_compressed(T, l, d)
    dXc = rng.standard_normal((Nc, dx))
    dX, dPE, _ = BW.compress_bwd(X, PE, W, l, d, dXc)
    ref = np.zeros((T, dx))
    for s in range(T):
        for i in range(Nc):
            if d * i <= s < d * i + l:
                ref[s] += dXc[i] / l
    np.testing.assert_allclose(dX, ref, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(dPE, np.broadcast_to(dXc.sum(axis=0) / l, (l, dx)), rtol=1e-13)


def test_key_shift_invariance_gives_zero_dpe_k(case):
    """Softmax is unchanged when one vector is added to every key of a branch
    (each score of a row moves by the same q . c), so the gradients of a
    branch's keys sum to zero for every query: sum_j dS_j = sum_j P_j (dP_j -
    dO . O) = dO . O - dO . O = 0.  Summed over the compressed cache this
    makes sum_i dKc_i = 0, hence dPE_K = sum_i dKc_i W_r^T = 0, while dPE_V
    (values carry no such invariance) is not."""
    inp, dout, idx, _ = case
    g = BW.nsa_prefill_backward(inp, dout, params=PARAMS, idx=idx)
    assert g["dkc"].shape[1] > 0
    scale_k = np.abs(g["dkc"]).sum(axis=1).max()
    assert np.abs(g["dkc"].sum(axis=1)).max() <= 1e-12 * scale_k
    assert np.abs(g["dpe_k"]).max() <= 1e-12 * np.abs(g["dw_k"]).max()
    assert np.abs(g["dpe_v"]).max() > 1e-3 * np.abs(g["dw_v"]).max()
    # selected and window keys: each row's gradient over its own keys sums to
    # zero too, so the token-level dk summed over all tokens (minus the part
    # that reaches the tokens through the compression map) vanishes
    K = BW._inputs_f64(inp, 0)["k"]
    for gg in range(WL.G):
        dKx, _, _ = BW.compress_bwd(K[:, gg], BW._inputs_f64(inp, 0)["pe_k"], BW._inputs_f64(inp, 0)["w_k"],
                                    PARAMS.l, PARAMS.d, g["dkc"][gg])
        direct = g["dk"][:, gg] - dKx
        assert np.abs(direct.sum(axis=0)).max() <= 1e-10 * np.abs(direct).sum(axis=0).max()


def test_combined_output_matches_an_independent_formulation(case):
    """The combined forward output (the three branches and the gates) of the
    forward oracle against the torch formulation above, on the same kept
    blocks and the same bf16-rounded cache: a dropped branch, a gate taken
    from the wrong column or a mis-masked branch would differ by O(1)."""
    inp, _, idx, x = case
    ref = O.nsa_prefill_reference(inp, params=PARAMS)
    xt = {kk: torch.tensor(vv, dtype=torch.float64) for kk, vv in x.items()}
    got = _torch_forward_out(xt, idx, round_cache=True).numpy()
    np.testing.assert_allclose(ref["out"], got, rtol=1e-10, atol=1e-12)
    # the per-branch outputs are mixed by the gates in the order (cmp, slc, win)
    g = x["gates"][..., None]
    np.testing.assert_allclose(ref["out"], g[:, :, 0] * ref["o_cmp"] + g[:, :, 1] * ref["o_slc"] +
                               g[:, :, 2] * ref["o_win"], rtol=1e-12, atol=1e-14)
