"""GPU parity of nsa_decode_step against the fp64 oracle (row t = T-1 of the
NSA forward, read from head-major caches).

Same rules as the prefill parity tests: kept block indices bit-exact except
near-ties (fp32 score gap at the cut below 1e-5 relative, where the GPU's set
must be one of the oracle's valid alternatives and the output is compared with
the oracle evaluated on that set); outputs within 2e-2 max and 2e-3 mean
absolute error.
"""
import math

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

from oracle import nsa as O
from workloads import DecodeWorkload, NSAParams, decode_config, make_decode
from tests.gpu_util import bf16_compare, cache_f64, compress_exact

MAX_ABS, MEAN_ABS, NEAR_TIE = 2e-2, 2e-3, 1e-5


def _nsa():
    import sparse_attention_long_10_b300 as nsa
    return nsa


def run_decode(inp, kc=None, vc=None, params=NSAParams(), idx_fill=-7, seq_lens=None, expect_status=0):
    """Decode through the C-ABI.  kc/vc: oracle compressed caches [B,G,Nc,d]
    (fp64 on the bf16 grid); when None the GPU compresses the caches itself
    with nsa_compress_kv (head-major layout)."""
    nsa = _nsa()
    d = {k: t.cuda() for k, t in inp.items()}
    B, G, T, dk = inp["kcache"].shape
    H = inp["q"].shape[1]
    dv = inp["vcache"].shape[3]
    cfg = nsa.make_cfg(B, T, H, G, dk, dv, phi=d, l=params.l, d=params.d, lsel=params.lsel,
                       n=params.n, w=params.w)
    Nc = nsa.nsa_num_compressed(cfg)
    if kc is not None:
        kc_t = torch.from_numpy(np.ascontiguousarray(kc)).to(torch.bfloat16).reshape(B, G, Nc, dk).cuda()
        vc_t = torch.from_numpy(np.ascontiguousarray(vc)).to(torch.bfloat16).reshape(B, G, Nc, dv).cuda()
    else:
        kc_t = torch.empty(B, G, Nc, dk, dtype=torch.bfloat16, device="cuda")
        vc_t = torch.empty(B, G, Nc, dv, dtype=torch.bfloat16, device="cuda")
        cws = nsa.workspace(nsa.nsa_compress_workspace_size(cfg))
        nsa.nsa_compress_kv(cfg, nsa.NSA_LAYOUT_BGTD, d["kcache"], d["vcache"], kc_t, vc_t, cws)
    out = torch.full((B, H, dv), float("nan"), dtype=torch.bfloat16, device="cuda")
    idx = torch.full((B, G, params.n), idx_fill, dtype=torch.int32, device="cuda")
    ws = nsa.workspace(nsa.nsa_decode_workspace_size(cfg))
    lens = None if seq_lens is None else torch.tensor(seq_lens, dtype=torch.int32, device="cuda")
    nsa.nsa_decode_step(cfg, d["q"], d["kcache"], d["vcache"], kc_t, vc_t, d["gates"], out, idx, ws,
                        seq_lens=lens)
    torch.cuda.synchronize()
    assert nsa.nsa_device_status(ws) == expect_status
    return out, idx, kc_t, vc_t


def check_decode(inp, ref, out, idx, params=NSAParams(), label="", near_tie=NEAR_TIE):
    """Compare the GPU result of the sequences ref['seqs'] with the oracle."""
    B, G, T, dk = inp["kcache"].shape
    H = inp["q"].shape[1]
    hpg = H // G
    scale = 1.0 / math.sqrt(dk)
    seqs = [int(s) for s in ref["seqs"]]
    lens = [int(x) for x in ref["lens"]]
    got = out[torch.as_tensor(seqs)].float().cpu().numpy()       # [S,H,dv]
    gidx = idx[torch.as_tensor(seqs)].cpu().numpy()              # [S,G,n]
    expect = ref["out"].copy()
    near = 0
    for si, b in enumerate(seqs):
        t = lens[si] - 1
        for g in range(G):
            if np.array_equal(gidx[si, g], ref["idx"][si, g]):
                continue
            ok, gap = O.selection_set_valid(ref["S32"][si, g], t, gidx[si, g], params.n, params.lsel, near_tie)
            assert ok, (f"{label} seq {b} g={g}: GPU blocks {gidx[si, g].tolist()} vs oracle "
                        f"{ref['idx'][si, g].tolist()} (gap {gap:.3g})")
            near += 1
            hs = slice(g * hpg, (g + 1) * hpg)
            q = O.to_f64(inp["q"][b, hs])
            K = O.to_f64(inp["kcache"][b, g, :t + 1])
            V = O.to_f64(inp["vcache"][b, g, :t + 1])
            o_slc = O.sel_attention(q, t, K, V, gidx[si, g], params.lsel, scale)
            gt = O.to_f64(inp["gates"][b, hs])
            expect[si, hs] = (gt[:, 0:1] * ref["o_cmp"][si, hs] + gt[:, 1:2] * o_slc
                              + gt[:, 2:3] * ref["o_win"][si, hs])
    assert np.isfinite(got).all(), f"{label}: non-finite output"
    err = np.abs(got - expect)
    print(f"{label}: seqs={len(seqs)} max_abs={err.max():.3e} mean_abs={err.mean():.3e} near_ties={near}")
    assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, label
    return near


TINY = DecodeWorkload("nsa_decode_tiny", 3, 2048, 4, 1, 64, 64, 5)
MID = DecodeWorkload("nsa_decode_mid", 2, 5000, 32, 2, 192, 128, 6)


@pytest.mark.parametrize("T", [2048, 1088, 1087, 1000, 1234, 97, 64, 65, 37, 32, 31, 1])
def test_decode_tiny_ragged(T):
    inp = make_decode(TINY, T=T)
    ref = O.nsa_decode_reference(inp)
    out, idx, _, _ = run_decode(inp, ref["kc"], ref["vc"])
    check_decode(inp, ref, out, idx, label=f"decode tiny T={T}")


@pytest.mark.parametrize("which,name", [(0, "cmp"), (1, "slc"), (2, "win")])
def test_decode_single_branch(which, name):
    inp = make_decode(TINY, T=3000)
    g = torch.zeros_like(inp["gates"])
    g[..., which] = 1.0
    inp["gates"] = g
    ref = O.nsa_decode_reference(inp)
    out, idx, _, _ = run_decode(inp, ref["kc"], ref["vc"])
    check_decode(inp, ref, out, idx, label=f"decode branch {name}")


def test_decode_mid_heads_and_dims():
    inp = make_decode(MID)
    ref = O.nsa_decode_reference(inp)
    out, idx, _, _ = run_decode(inp, ref["kc"], ref["vc"])
    check_decode(inp, ref, out, idx, label="decode mid")


def test_decode_end_to_end_compression():
    # the GPU compresses the caches; its cache is checked against the exact
    # compression, then the oracle scores that same cache (strict near-ties)
    inp = make_decode(MID)
    out, idx, kc, vc = run_decode(inp)
    B, G = MID.B, MID.G
    bf16_compare(kc, *compress_exact(inp, B, G, False, "kcache", "pe_k", "w_k"))
    bf16_compare(vc, *compress_exact(inp, B, G, False, "vcache", "pe_v", "w_v"))
    ref = O.nsa_decode_reference(inp, kc=cache_f64(kc), vc=cache_f64(vc))
    check_decode(inp, ref, out, idx, label="decode end-to-end")


RAGGED = DecodeWorkload("nsa_decode_ragged", 7, 5000, 32, 2, 192, 128, 8)


def test_decode_ragged_batch_lengths():
    """One batch whose sequences have different lengths (seq_lens): each
    query sits at its own len-1 and reads only its own tokens."""
    inp = make_decode(RAGGED)
    lens = [1, 31, 64, 1087, 2048, 5000, 4999]
    ref = O.nsa_decode_reference(inp, seq_lens=lens)
    out, idx, _, _ = run_decode(inp, ref["kc"], ref["vc"], seq_lens=lens)
    check_decode(inp, ref, out, idx, label="decode ragged")


def test_decode_ragged_end_to_end_compression():
    # the GPU compresses the caches at capacity; each sequence uses its prefix
    inp = make_decode(RAGGED)
    lens = [5000, 97, 4096, 4097, 600, 33, 1]
    out, idx, kc, vc = run_decode(inp, seq_lens=lens)
    ref = O.nsa_decode_reference(inp, kc=cache_f64(kc), vc=cache_f64(vc), seq_lens=lens)
    check_decode(inp, ref, out, idx, label="decode ragged end-to-end")


def test_decode_invalid_lengths_are_reported_and_skipped():
    """Lengths outside [1, T] are read on the device: the step records
    NSA_ERR_INVALID_ARG, reads nothing of those sequences (output zero, no
    kept blocks) and computes the valid ones as usual."""
    inp = make_decode(RAGGED)
    T = RAGGED.T
    lens = [0, 2048, -3, T + 1, 777, T, 1 << 30]
    out, idx, kc, vc = run_decode(inp, seq_lens=lens, expect_status=1)   # 1 = NSA_ERR_INVALID_ARG
    bad = torch.as_tensor([0, 2, 3, 6])
    assert torch.all(out[bad].float() == 0) and torch.all(idx[bad] == -1)
    good = [1, 4, 5]
    ref = O.nsa_decode_reference(inp, seqs=good, kc=cache_f64(kc), vc=cache_f64(vc),
                                 seq_lens=[L if 1 <= L <= T else T for L in lens])
    check_decode(inp, ref, out, idx, label="decode with invalid lengths")


def test_decode_twice_is_deterministic():
    inp = make_decode(MID)
    out1, idx1, _, _ = run_decode(inp)
    out2, idx2, _, _ = run_decode(inp)
    assert torch.equal(idx1, idx2)
    assert torch.equal(out1, out2)


def test_decode_full_size_all_sequences():
    """The 16 x 65,536-token decode step in the launch configuration the
    benchmark times (GPU compression of the caches, then the step).  Every
    sequence's compressed cache is checked against the exact compression, and
    the oracle, scoring that same cache, checks all sixteen sequences."""
    wl = decode_config()
    inp = make_decode(wl)
    out, idx, kc, vc = run_decode(inp)
    for b0 in range(0, wl.B, 4):
        seqs = list(range(b0, b0 + 4))
        ek, mk = compress_exact(inp, wl.B, wl.G, False, "kcache", "pe_k", "w_k", seqs=seqs)
        bf16_compare(kc[b0:b0 + 4], ek, mk)
        ev, mv = compress_exact(inp, wl.B, wl.G, False, "vcache", "pe_v", "w_v", seqs=seqs)
        bf16_compare(vc[b0:b0 + 4], ev, mv)
    ref = O.nsa_decode_reference(inp, kc=cache_f64(kc), vc=cache_f64(vc))
    check_decode(inp, ref, out, idx, label="decode 16x64k")
