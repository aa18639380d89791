"""GPU parity of dsa_decode_step against the fp64 oracle (indexer scores,
top-k positions with ties to the lower position, attention over the kept set
only).

Rules: kept positions bit-exact except where the fp32 score gap at the cut is
below 1e-5 relative (near-ties: the GPU set must keep every position clearly
above the cut and take the rest from the band at the cut; the output is then
compared with the oracle evaluated on the GPU's set); outputs within 2e-2 max
and 2e-3 mean absolute error.
"""
import math

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

from oracle import dsa as D
from oracle import nsa as O
from workloads import DSAWorkload, dsa_config, make_dsa

MAX_ABS, MEAN_ABS, NEAR_TIE = 2e-2, 2e-3, 1e-5


def _nsa():
    import sparse_attention_long_10_b300 as nsa
    return nsa


def run_dsa(inp, topk, latent_dv=None, seq_lens=None, expect_status=0):
    """inp["v"] None: latent values, the first latent_dv columns of k.
    seq_lens: per-row context lengths (device int32), None for all T."""
    nsa = _nsa()
    d = {k: t.cuda() for k, t in inp.items() if t is not None}
    B, T, dI = inp["kI"].shape
    HI = inp["qI"].shape[1]
    H, dk = inp["q"].shape[1], inp["q"].shape[2]
    dv = inp["v"].shape[2] if inp.get("v") is not None else latent_dv
    cfg = nsa.make_dsa_cfg(B, T, HI, dI, H, dk, dv, topk)
    kk = min(topk, T)
    out = torch.full((B, H, dv), float("nan"), dtype=torch.bfloat16, device="cuda")
    idx = torch.full((B, kk), -7, dtype=torch.int32, device="cuda")
    ws = nsa.workspace(nsa.dsa_decode_workspace_size(cfg))
    lens = None if seq_lens is None else torch.tensor(seq_lens, dtype=torch.int32, device="cuda")
    nsa.dsa_decode_step(cfg, d["qI"], d["wI"], d["kI"], d["q"], d["k"], d.get("v"), out, idx, ws, seq_lens=lens)
    torch.cuda.synchronize()
    assert nsa.nsa_device_status(ws) == expect_status
    return out, idx


def check_dsa(inp, ref, out, idx, topk, label="", exact_idx=False):
    batches = [int(b) for b in ref["batches"]]
    dk = inp["q"].shape[2]
    scale = 1.0 / math.sqrt(dk)
    got = out[torch.as_tensor(batches)].float().cpu().numpy()
    gidx = idx[torch.as_tensor(batches)].cpu().numpy()
    expect = ref["out"].copy()
    near = 0
    lens = [int(x) for x in ref["lens"]]
    for si, b in enumerate(batches):
        Tb = lens[si]
        kk = min(topk, Tb)
        assert (gidx[si, kk:] == -1).all(), f"{label} b={b}: -1 padding past the kept positions"
        row = gidx[si, :kk]
        assert list(row) == sorted(set(row.tolist())), f"{label} b={b}: positions not ascending/distinct"
        if np.array_equal(row, ref["idx"][si, :kk]):
            continue
        assert not exact_idx, f"{label} b={b}: kept set differs from the oracle's"
        ok, gap = D.topk_set_valid(ref["I32"][si, :Tb], row, topk, NEAR_TIE)
        assert ok, f"{label} b={b}: GPU set is not a valid top-{topk} (gap {gap:.3g})"
        near += 1
        ti = torch.as_tensor(row.astype(np.int64))
        Ksel = O.to_f64(inp["k"][b, ti])
        Vsel = Ksel[:, :expect.shape[2]] if inp.get("v") is None else O.to_f64(inp["v"][b, ti])
        expect[si] = D.dsa_attention(O.to_f64(inp["q"][b]), Ksel, Vsel, scale)
    assert np.isfinite(got).all(), f"{label}: non-finite output"
    err = np.abs(got - expect)
    print(f"{label}: rows={len(batches)} max_abs={err.max():.3e} mean_abs={err.mean():.3e} near_ties={near}")
    assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, label


SMALL = DSAWorkload("dsa_small", 2, 3000, 4, 64, 16, 576, 512, 256, 7)
DIMS = DSAWorkload("dsa_dims", 3, 5000, 2, 128, 4, 128, 64, 300, 8)


@pytest.mark.parametrize("T,topk", [(3000, 256), (3000, 2048), (4097, 2048), (1000, 1), (1000, 7),
                                    (2049, 2049), (700, 2048), (1, 5)])
def test_dsa_small(T, topk):
    inp = make_dsa(SMALL, T=T)
    ref = D.dsa_decode_reference(inp, topk)
    out, idx = run_dsa(inp, topk)
    check_dsa(inp, ref, out, idx, topk, label=f"dsa T={T} k={topk}")


def test_dsa_other_dims():
    inp = make_dsa(DIMS)
    ref = D.dsa_decode_reference(inp, DIMS.topk)
    out, idx = run_dsa(inp, DIMS.topk)
    check_dsa(inp, ref, out, idx, DIMS.topk, label="dsa dims")


def test_dsa_exact_ties_go_to_lower_positions():
    # negative indexer weights: every score is <= 0 and the positions whose
    # indexer dot products are all <= 0 score exactly 0 -- the best value --
    # so the top-k is decided among exact ties by position alone
    inp = make_dsa(SMALL, T=4096)
    inp["wI"] = -torch.ones_like(inp["wI"])
    ref = D.dsa_decode_reference(inp, 100)
    assert all((ref["I32"][r][ref["idx"][r]] == 0).all() for r in range(SMALL.B))
    out, idx = run_dsa(inp, 100)
    check_dsa(inp, ref, out, idx, 100, label="dsa exact ties", exact_idx=True)


def test_dsa_all_equal_scores_use_the_slow_resolve():
    # zero weights: all 20000 scores equal, more boundary candidates than the
    # candidate buffer holds; the kept set must be the 5000 lowest positions
    inp = make_dsa(SMALL, T=20000)
    inp["wI"] = torch.zeros_like(inp["wI"])
    ref = D.dsa_decode_reference(inp, 5000)
    np.testing.assert_array_equal(ref["idx"][0], np.arange(5000))
    out, idx = run_dsa(inp, 5000)
    check_dsa(inp, ref, out, idx, 5000, label="dsa all equal", exact_idx=True)


def test_dsa_full_size():
    """Batch 8 x 131,072-token context, top-2048: the configuration the
    benchmark times; the oracle checks every row."""
    wl = dsa_config()
    inp = make_dsa(wl)
    out, idx = run_dsa(inp, wl.topk)
    ref = D.dsa_decode_reference(inp, wl.topk)
    check_dsa(inp, ref, out, idx, wl.topk, label="dsa 8x128k")


def test_dsa_twice_is_deterministic():
    inp = make_dsa(SMALL)
    o1, i1 = run_dsa(inp, 256)
    o2, i2 = run_dsa(inp, 256)
    assert torch.equal(i1, i2) and torch.equal(o1, o2)


@pytest.mark.parametrize("T,topk", [(3000, 256), (3000, 2048), (700, 2048), (1, 5)])
def test_dsa_latent_values_small(T, topk):
    """Latent KV: values are the first dv columns of the key rows (v = NULL)."""
    inp = make_dsa(SMALL, T=T)
    inp["v"] = None
    ref = D.dsa_decode_reference(inp, topk, latent_dv=SMALL.dv)
    out, idx = run_dsa(inp, topk, latent_dv=SMALL.dv)
    check_dsa(inp, ref, out, idx, topk, label=f"dsa latent T={T} k={topk}")


def test_dsa_latent_values_full_size():
    """Batch 8 x 131,072-token context, top-2048, dk=576 latent keys whose
    first 512 columns are the values; the oracle checks every row."""
    wl = dsa_config()
    inp = make_dsa(wl)
    inp["v"] = None
    out, idx = run_dsa(inp, wl.topk, latent_dv=wl.dv)
    ref = D.dsa_decode_reference(inp, wl.topk, latent_dv=wl.dv)
    check_dsa(inp, ref, out, idx, wl.topk, label="dsa latent 8x128k")


def test_dsa_rows_with_different_lengths():
    """One batch whose rows hold different context lengths (seq_lens): each
    row scores and keeps among its own positions only."""
    wl = DSAWorkload("dsa_ragged", 6, 5000, 4, 64, 16, 576, 512, 256, 17)
    inp = make_dsa(wl)
    lens = [5000, 1, 255, 256, 257, 3001]
    ref = D.dsa_decode_reference(inp, wl.topk, seq_lens=lens)
    out, idx = run_dsa(inp, wl.topk, seq_lens=lens)
    check_dsa(inp, ref, out, idx, wl.topk, label="dsa ragged")


def test_dsa_invalid_lengths_are_reported_and_skipped():
    wl = DSAWorkload("dsa_ragged_bad", 4, 3000, 4, 64, 16, 576, 512, 256, 18)
    inp = make_dsa(wl)
    lens = [0, 3000, 3001, 700]
    out, idx = run_dsa(inp, wl.topk, seq_lens=lens, expect_status=1)   # 1 = NSA_ERR_INVALID_ARG
    bad = torch.as_tensor([0, 2])
    assert torch.all(out[bad].float() == 0) and torch.all(idx[bad] == -1)
    ref = D.dsa_decode_reference(inp, wl.topk, batches=[1, 3], seq_lens=[3000, 3000, 3000, 700])
    check_dsa(inp, ref, out, idx, wl.topk, label="dsa with invalid lengths")
