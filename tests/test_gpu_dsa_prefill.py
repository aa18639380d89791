"""GPU parity of dsa_prefill_fwd (every position a query) against the fp64
oracle ``oracle.dsa.dsa_prefill_reference``: row t scores and keeps among its
causal prefix s <= t, min(topk, t+1) positions, ties to the lower position,
and attends over them.

Rules as for the decode step: kept positions bit-exact except at fp32 near
ties (gap below 1e-5 relative at the cut: the GPU set must be a valid top-k,
and its output is compared with the oracle evaluated on the GPU's set);
outputs within 2e-2 max and 2e-3 mean absolute error.
"""
import math

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

from oracle import dsa as D
from oracle import nsa as O
from workloads import DSAWorkload, dsa_prefill_config, make_dsa_prefill

MAX_ABS, MEAN_ABS, NEAR_TIE = 2e-2, 2e-3, 1e-5


def _nsa():
    import sparse_attention_long_10_b300 as nsa
    return nsa


def run_prefill(inp, topk, latent_dv=None):
    """inp["v"] None: latent values, the first latent_dv columns of k."""
    nsa = _nsa()
    d = {k: t.cuda() for k, t in inp.items() if t is not None}
    B, T, dI = inp["kI"].shape
    HI = inp["qI"].shape[2]
    H, dk = inp["q"].shape[2], inp["q"].shape[3]
    dv = inp["v"].shape[2] if inp.get("v") is not None else latent_dv
    cfg = nsa.make_dsa_cfg(B, T, HI, dI, H, dk, dv, topk)
    kk = min(topk, T)
    out = torch.full((B, T, H, dv), float("nan"), dtype=torch.bfloat16, device="cuda")
    idx = torch.full((B, T, kk), -7, dtype=torch.int32, device="cuda")
    ws = nsa.workspace(nsa.dsa_prefill_workspace_size(cfg))
    nsa.dsa_prefill_fwd(cfg, d["qI"], d["wI"], d["kI"], d["q"], d["k"], d.get("v"), out, idx, ws)
    torch.cuda.synchronize()
    assert nsa.nsa_device_status(ws) == 0
    return out, idx


def check_rows(inp, out, idx, topk, b, rows, label="", exact_idx=False, latent_dv=None):
    ref_inp = dict(inp)
    if inp.get("v") is None:
        ref_inp["v"] = inp["k"][..., :latent_dv].contiguous()
    ref = D.dsa_prefill_reference(ref_inp, topk, b=b, rows=rows)
    dk = inp["q"].shape[3]
    scale = 1.0 / math.sqrt(dk)
    rows_t = torch.as_tensor(list(rows))
    got = out[b, rows_t].float().cpu().numpy()
    gidx = idx[b, rows_t].cpu().numpy()
    expect = ref["out"].copy()
    near = 0
    for r, t in enumerate(rows):
        kk = min(topk, t + 1)
        assert (gidx[r, kk:] == -1).all(), f"{label} t={t}: -1 padding past the kept positions"
        row = gidx[r, :kk]
        if np.array_equal(row, ref["idx"][r]):
            continue
        assert not exact_idx, f"{label} t={t}: kept set differs from the oracle's"
        assert list(row) == sorted(set(row.tolist())), f"{label} t={t}: positions not ascending/distinct"
        ok, gap = D.topk_set_valid(ref["I32"][r], row, topk, NEAR_TIE)
        assert ok, f"{label} t={t}: GPU set is not a valid top-{topk} (gap {gap:.3g})"
        near += 1
        ti = torch.as_tensor(row.astype(np.int64))
        Ksel = O.to_f64(ref_inp["k"][b, ti])
        Vsel = O.to_f64(ref_inp["v"][b, ti])
        expect[r] = D.dsa_attention(O.to_f64(inp["q"][b, t]), Ksel, Vsel, scale)
    assert np.isfinite(got).all(), f"{label}: non-finite output"
    err = np.abs(got - expect)
    print(f"{label}: rows={len(rows)} max_abs={err.max():.3e} mean_abs={err.mean():.3e} near_ties={near}")
    assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, label


SMALL = DSAWorkload("dsa_prefill_small", 2, 700, 4, 64, 16, 128, 64, 256, 11)
LATENT = DSAWorkload("dsa_prefill_latent", 1, 400, 4, 64, 16, 576, 512, 128, 12)
BENCH = dsa_prefill_config()


def test_dsa_prefill_every_row():
    """Both sequences, every row: rows t < 256 keep their whole prefix, the
    later ones a top-256."""
    inp = make_dsa_prefill(SMALL)
    out, idx = run_prefill(inp, SMALL.topk)
    for b in range(SMALL.B):
        check_rows(inp, out, idx, SMALL.topk, b, range(SMALL.T), label=f"dsa prefill b={b}")


def test_dsa_prefill_latent_values():
    inp = make_dsa_prefill(LATENT)
    inp["v"] = None
    out, idx = run_prefill(inp, LATENT.topk, latent_dv=LATENT.dv)
    check_rows(inp, out, idx, LATENT.topk, 0, range(LATENT.T), label="dsa prefill latent",
               latent_dv=LATENT.dv)


def test_dsa_prefill_topk_covers_every_prefix_is_causal_attention():
    inp = make_dsa_prefill(SMALL, B=1, T=300)
    out, idx = run_prefill(inp, 512)
    check_rows(inp, out, idx, 512, 0, range(300), label="dsa prefill full causal", exact_idx=True)
    kk = idx[0].cpu().numpy()
    for t in (0, 1, 150, 299):
        np.testing.assert_array_equal(kk[t, :t + 1], np.arange(t + 1))


def test_dsa_prefill_exact_ties_go_to_lower_positions():
    # negative indexer weights: positions whose indexer dot products are all
    # <= 0 score exactly 0, the best value, so ties are decided by position
    inp = make_dsa_prefill(SMALL, B=1, T=600)
    inp["wI"] = -torch.ones_like(inp["wI"])
    out, idx = run_prefill(inp, 50)
    check_rows(inp, out, idx, 50, 0, range(600), label="dsa prefill exact ties", exact_idx=True)


def test_dsa_prefill_bench_shape_sampled_rows():
    """The benchmark's shape (one 8192-token sequence, latent 576/512 keys,
    top-2048): 96 rows spread over the sequence plus the last 8."""
    inp = make_dsa_prefill(BENCH)
    inp["v"] = None
    out, idx = run_prefill(inp, BENCH.topk, latent_dv=BENCH.dv)
    rng = np.random.default_rng(5)
    rows = sorted(set(rng.integers(0, BENCH.T, 96).tolist()) | set(range(BENCH.T - 8, BENCH.T)) | {0, 2047, 2048})
    check_rows(inp, out, idx, BENCH.topk, 0, rows, label="dsa prefill 8192", latent_dv=BENCH.dv)


def test_dsa_prefill_twice_is_deterministic():
    inp = make_dsa_prefill(SMALL, B=1)
    o1, i1 = run_prefill(inp, 100)
    o2, i2 = run_prefill(inp, 100)
    assert torch.equal(i1, i2) and torch.equal(o1, o2)
