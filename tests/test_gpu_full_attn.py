"""GPU parity of nsa_full_attn_fwd (exact causal full attention, the dense
comparison of the benchmark) against the oracle's attention over s <= t.

The oracle's window attention with a window covering the whole prefix is
causal full attention (pinned on the CPU by the textbook-softmax reduction
tests).  Tolerances: 2e-2 max and 2e-3 mean absolute error (bf16 inputs, fp32
accumulation, bf16 output)."""
import math

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

from oracle import nsa as O
from workloads import PREFILL_CONFIGS, make_prefill

MAX_ABS, MEAN_ABS = 2e-2, 2e-3


def run_full(inp):
    import sparse_attention_long_10_b300 as nsa
    d = {k: inp[k].cuda() for k in ("q", "k", "v")}
    B, T, H, dk = inp["q"].shape
    G, dv = inp["k"].shape[2], inp["v"].shape[3]
    cfg = nsa.make_cfg(B, T, H, G, dk, dv)
    out = torch.full((B, T, H, dv), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = nsa.workspace(nsa.nsa_full_attn_workspace_size(cfg))
    nsa.nsa_full_attn_fwd(cfg, d["q"], d["k"], d["v"], out, ws)
    torch.cuda.synchronize()
    assert nsa.nsa_device_status(ws) == 0
    return out


def check(inp, out, rows, b=0, label=""):
    B, T, H, dk = inp["q"].shape
    G = inp["k"].shape[2]
    hpg = H // G
    scale = 1.0 / math.sqrt(dk)
    got = out[b, torch.as_tensor(rows)].float().cpu().numpy()
    ref = np.zeros_like(got, dtype=np.float64)
    for g in range(G):
        K = O.to_f64(inp["k"][b, :, g])
        V = O.to_f64(inp["v"][b, :, g])
        hs = slice(g * hpg, (g + 1) * hpg)
        for r, t in enumerate(rows):
            ref[r, hs] = O.win_attention(O.to_f64(inp["q"][b, t, hs]), int(t), K, V, T + 1, scale)
    assert np.isfinite(got).all(), label
    err = np.abs(got - ref)
    print(f"{label}: rows={len(rows)} max_abs={err.max():.3e} mean_abs={err.mean():.3e}")
    assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, label


@pytest.mark.parametrize("T", [2048, 1000, 129, 97, 1])
def test_full_attention_tiny_all_rows(T):
    wl = PREFILL_CONFIGS["tiny_2k"]
    inp = make_prefill(wl, T=T)
    out = run_full(inp)
    check(inp, out, list(range(T)), label=f"full tiny T={T}")


def test_full_attention_8k_sampled_rows():
    wl = PREFILL_CONFIGS["prefill_8k"]
    inp = make_prefill(wl)
    out = run_full(inp)
    rng = np.random.default_rng(21)
    rows = sorted(set([0, 1, 7, 8, 127, 128, 4095, wl.T - 8, wl.T - 1] + rng.integers(0, wl.T, 60).tolist()))
    check(inp, out, rows, label="full 8k")


def test_full_attention_64k_sampled_rows():
    """The dense comparison at the benchmark's 65,536-token size: rows spread
    over the sequence (the longest rows attend to every earlier token)."""
    wl = PREFILL_CONFIGS["prefill_64k"]
    inp = make_prefill(wl)
    out = run_full(inp)
    rng = np.random.default_rng(22)
    rows = sorted(set([0, 7, 8, 32767, wl.T - 2, wl.T - 1] + rng.integers(0, wl.T, 26).tolist()))
    check(inp, out, rows, label="full 64k")
