"""GPU parity of nsa_prefill_bwd against the fp64 backward oracle
``oracle.nsa_bwd.nsa_prefill_backward``.

The GPU forward runs first, on the oracle's bf16 compressed cache
(NSA_FLAG_KC_GIVEN), and hands that cache and its kept blocks to the
backward; the oracle computes its own forward selection, which must equal
the GPU's (bit-exact kept blocks).  Both sides therefore attend to the same
bf16 keys and values.

Tolerances, from the arithmetic: the backward's inputs are bf16 and every
contraction accumulates in fp32, but P * g and dS are rounded to bf16 (a
relative error of at most 2^-9 per term) before the dV, dK and dq
contractions, as the forward rounds P.  Each gradient tensor X is compared
by its own scale:
    max |gpu - ref| <= 1e-2 * max |ref|,
    mean |gpu - ref| <= 3e-3 * mean |ref|   (about 1.5 x 2^-9: one bf16
                                            rounding of every term of the sums);
dgates = dout . O_b has no bf16 step (fp32 scores, exponentials and sums):
1e-4 * max |ref|.
"""
import math

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

from oracle import nsa as O
from oracle import nsa_bwd as BW
from workloads import NSAParams, PrefillWorkload, make_prefill, make_prefill_dout

REL_MAX, REL_MEAN, REL_MAX_GATES = 1e-2, 3e-3, 1e-4
GRADS = ("dq", "dk", "dv", "dgates", "dw_k", "dw_v", "dpe_k", "dpe_v")


def _nsa():
    import sparse_attention_long_10_b300 as nsa
    return nsa


def oracle_cache(inp):
    """The oracle's bf16-rounded compressed cache [B,G,Nc,d] of K and of V."""
    B, T, G, _ = inp["k"].shape
    out = []
    for name, pe, w in (("k", "pe_k", "w_k"), ("v", "pe_v", "w_v")):
        pe64, w64 = O.to_f64(inp[pe]), O.to_f64(inp[w])
        out.append(np.stack([np.stack([O.compress(O.to_f64(inp[name][b, :, g]), pe64, w64, 32, 16)
                                       for g in range(G)]) for b in range(B)]))
    return out


def run_fwd_bwd(inp, dout, params=NSAParams(), caches=None, saved=False):
    """saved: the forward saves the selected branch's statistics
    (nsa_prefill_fwd_train) and the backward reads them."""
    nsa = _nsa()
    d = {k: t.cuda() for k, t in inp.items()}
    B, T, H, dk = inp["q"].shape
    G, dv = inp["k"].shape[2], inp["v"].shape[3]
    cfg = nsa.make_cfg(B, T, H, G, dk, dv, phi=d, l=params.l, d=params.d, lsel=params.lsel, n=params.n,
                       w=params.w, flags=nsa.NSA_FLAG_KC_GIVEN)
    Nc = nsa.nsa_num_compressed(cfg)
    if Nc > 0:
        kc64, vc64 = caches if caches is not None else oracle_cache(inp)
        kc = torch.from_numpy(kc64).to(torch.bfloat16).cuda()
        vc = torch.from_numpy(vc64).to(torch.bfloat16).cuda()
    else:
        kc = torch.empty(B, G, 1, dk, dtype=torch.bfloat16, device="cuda")
        vc = torch.empty(B, G, 1, dv, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(B, T, H, dv, dtype=torch.bfloat16, device="cuda")
    idx = torch.full((B, T, G, params.n), -7, dtype=torch.int32, device="cuda")
    ws = nsa.workspace(nsa.nsa_prefill_workspace_size(cfg))
    f32 = dict(device="cuda", dtype=torch.float32)
    lse = o = None
    if saved:
        lse = torch.full((B, T, H), float("nan"), **f32)
        o = torch.full((B, T, H, dv), float("nan"), **f32)
        nsa.nsa_prefill_fwd_train(cfg, d["q"], d["k"], d["v"], d["gates"], kc, vc, out, idx, lse, o, ws)
    else:
        nsa.nsa_prefill_fwd(cfg, d["q"], d["k"], d["v"], d["gates"], kc, vc, out, idx, ws)
    g = dict(dq=torch.full((B, T, H, dk), float("nan"), **f32), dk=torch.full((B, T, G, dk), float("nan"), **f32),
             dv=torch.full((B, T, G, dv), float("nan"), **f32), dgates=torch.full((B, T, H, 3), float("nan"), **f32),
             dw_k=torch.full((32 * dk, dk), float("nan"), **f32), dw_v=torch.full((32 * dv, dv), float("nan"), **f32),
             dpe_k=torch.full((32, dk), float("nan"), **f32), dpe_v=torch.full((32, dv), float("nan"), **f32))
    wsb = nsa.workspace(nsa.nsa_prefill_bwd_workspace_size(cfg))
    nsa.nsa_prefill_bwd(cfg, d["q"], d["k"], d["v"], d["gates"], kc, vc, idx, dout.cuda(), g["dq"], g["dk"],
                        g["dv"], g["dgates"], g["dw_k"], g["dw_v"], g["dpe_k"], g["dpe_v"], wsb, slc_lse=lse, slc_o=o)
    torch.cuda.synchronize()
    assert nsa.nsa_device_status(ws) == 0
    assert nsa.nsa_device_status(wsb) == 0
    return {k: v.cpu().numpy().astype(np.float64) for k, v in g.items()}, idx.cpu().numpy()


def compare(name, got, ref, label, scale=None, lim=None):
    """``scale``: the magnitude to measure errors against when the reference
    itself cancels to (near) zero."""
    assert np.isfinite(got).all(), f"{label} {name}: non-finite values"
    err = np.abs(got - ref)
    mx, mn = float(np.abs(ref).max()), float(np.abs(ref).mean())
    if scale is not None:
        mx, mn = float(np.abs(scale).max()), float(np.abs(scale).mean())
    rel_max = float(err.max()) / mx if mx > 0 else float(err.max())
    rel_mean = float(err.mean()) / mn if mn > 0 else float(err.mean())
    print(f"{label} {name}: max|ref|={mx:.3e} rel_max={rel_max:.2e} rel_mean={rel_mean:.2e}")
    if lim is None:
        lim = REL_MAX_GATES if name == "dgates" else REL_MAX
    assert rel_max <= lim, f"{label} {name}: rel max error {rel_max:.3e} > {lim}"
    assert rel_mean <= REL_MEAN, f"{label} {name}: rel mean error {rel_mean:.3e} > {REL_MEAN}"


def check_dgates(got, ref, label, saved):
    """With the forward's saved statistics the selected branch's dgates is
    dout . O_slc, where O_slc was formed with the forward's bf16 P (a 2^-9
    relative rounding of each term): that column is held to 2^-9."""
    if saved:
        compare("dgates[cmp,win]", got[..., [0, 2]], ref[..., [0, 2]], label, lim=REL_MAX_GATES)
        compare("dgates[slc]", got[..., 1], ref[..., 1], label, lim=2.0 ** -9)
    else:
        compare("dgates", got, ref, label)


def check_case(wl, label, T=None, saved=False):
    inp = make_prefill(wl, T=T)
    dout = make_prefill_dout(wl, T=T)
    got, gidx = run_fwd_bwd(inp, dout, wl.params, saved=saved)
    B = inp["q"].shape[0]
    acc = {k: np.zeros_like(got[k]) for k in ("dw_k", "dw_v", "dpe_k", "dpe_v")}
    # dPE_K = (sum_i dKc_i) W_r^T cancels to zero (softmax is invariant to a
    # shift of every key), so its error is measured against the size of the
    # uncancelled terms, sum_e (sum_i |dKc_i,e|) |W[r dk + c, e]|
    dk = inp["q"].shape[3]
    absw = np.abs(O.to_f64(inp["w_k"])).reshape(32, dk, dk)
    pe_scale = np.zeros((32, dk))
    for b in range(B):
        ref = BW.nsa_prefill_backward(inp, O.to_f64(dout[b]), b=b, params=wl.params)
        assert np.array_equal(gidx[b], ref["idx"]), f"{label} b={b}: kept blocks differ from the oracle's"
        for name in ("dq", "dk", "dv"):
            compare(name, got[name][b], ref[name], f"{label} b={b}")
        check_dgates(got["dgates"][b], ref["dgates"], f"{label} b={b}", saved)
        for k in acc:
            acc[k] += ref[k]
        if ref["dkc"].shape[1]:
            pe_scale += absw @ np.abs(ref["dkc"]).sum(axis=(0, 1))
    for k in acc:
        compare(k, got[k], acc[k], label, scale=pe_scale if k == "dpe_k" else None)


# one group of the benchmark's shapes (16 heads per group, dk 192, dv 128), a ragged tail
def test_backward_bench_group_shapes():
    wl = PrefillWorkload("bwd_T1000_H16_G1_dk192_dv128", 1, 1000, 16, 1, 192, 128, 21)
    check_case(wl, "bwd T=1000 dk192")


def test_backward_with_saved_forward_statistics():
    wl = PrefillWorkload("bwd_T1000_H16_G1_dk192_dv128", 1, 1000, 16, 1, 192, 128, 21)
    check_case(wl, "bwd saved T=1000 dk192", saved=True)


def test_backward_saved_statistics_batch_few_heads():
    wl = PrefillWorkload("bwd_B2_T700_H8_G2", 2, 700, 8, 2, 128, 128, 23, NSAParams(n=4, w=96))
    check_case(wl, "bwd saved B=2 hpg=4", saved=True)


def test_backward_two_groups_dk128_dv64():
    wl = PrefillWorkload("bwd_T1500_H32_G2_dk128_dv64", 1, 1500, 32, 2, 128, 64, 22)
    check_case(wl, "bwd T=1500 G=2")


def test_backward_batch_few_heads_short_window():
    # 4 heads per group (MMA columns padded to 16), two sequences, w = 96,
    # n = 4: a real top-n choice from block 4 on
    wl = PrefillWorkload("bwd_B2_T700_H8_G2", 2, 700, 8, 2, 128, 128, 23, NSAParams(n=4, w=96))
    check_case(wl, "bwd B=2 hpg=4")


@pytest.mark.parametrize("T", [20, 31, 32, 47, 130])
def test_backward_short_sequences(T):
    # T < 32: no compressed block at all; 32 / 47: one; 130: the first rows'
    # compressed branch is empty
    wl = PrefillWorkload(f"bwd_T{T}", 1, T, 16, 1, 128, 64, 24)
    check_case(wl, f"bwd T={T}")


def test_backward_full_size_sampled_rows():
    """The 64k benchmark shape (B=1, H=64, G=4, dk=192, dv=128), run as the
    benchmark runs it (the forward saves the selected branch's statistics):
    dq and dgates of 24 sampled rows per group against the oracle's per-row
    backward (the rows' own kept blocks from the oracle forward); dk, dv and
    the parameter gradients must be finite."""
    from workloads import PREFILL_CONFIGS
    wl = PREFILL_CONFIGS["prefill_64k"]
    inp = make_prefill(wl)
    dout = make_prefill_dout(wl)
    kc64, vc64 = oracle_cache(inp)
    got, gidx = run_fwd_bwd(inp, dout, wl.params, caches=(kc64, vc64), saved=True)
    for k in ("dk", "dv", "dw_k", "dw_v", "dpe_k", "dpe_v"):
        assert np.isfinite(got[k]).all(), k
    x = BW._inputs_f64(inp, 0)
    T, H, dk = x["q"].shape
    G = x["k"].shape[1]
    hpg = H // G
    scale = 1.0 / math.sqrt(dk)
    rng = np.random.default_rng(9)
    rows = np.array(sorted(set(rng.integers(0, T, 20).tolist()) | {0, 31, 4000, T - 1}))
    dout64 = O.to_f64(dout[0])
    for g in range(G):
        K, V = x["k"][:, g], x["v"][:, g]
        Kc, Vc = kc64[0, g], vc64[0, g]
        hs = slice(g * hpg, (g + 1) * hpg)
        fw = O.nsa_group_rows(x["q"][rows][:, hs], rows, K, V, Kc, Vc, x["gates"][rows][:, hs], wl.params, scale)
        assert np.array_equal(gidx[0, rows, g], fw["idx"]), f"g={g}: kept blocks differ"
        r = BW.nsa_group_bwd(x["q"][rows][:, hs], rows, K, V, Kc, Vc, x["gates"][rows][:, hs], fw["idx"],
                             wl.params, scale, dout64[rows][:, hs])
        compare("dq", got["dq"][0, rows][:, hs], r["dq"], f"64k g={g}")
        check_dgates(got["dgates"][0, rows][:, hs], r["dgates"], f"64k g={g}", True)
